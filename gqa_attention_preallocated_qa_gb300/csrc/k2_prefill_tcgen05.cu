// k2_prefill_tcgen05.cu -- K2: causal grouped-query flash attention over the
// prompt (prefill), on the 5th-generation tensor cores.
//
// "Prefill ... is a large share of total time" for prompts of 512-2048 tokens
// and 32-128 generated tokens (dryft-flash-infer agent guide, "Where the wins
// are", prefill bullet).  The result is exact causal softmax attention; only
// the order of the arithmetic differs from the definition ("reorderings are
// affordable", same guide, "Numerics").
//
// Two persistent forms walk fixed shares of the work items.  An item is one
// 128-row block of a sequence's new tokens (a whole prompt, or a chunk appended
// after the tokens the layer already holds) for some query heads of a kv head,
// all of which share every K/V tile: in the one-CTA form (one CTA per SM) one
// or two heads, in the CTA-pair form (two SMs, tcgen05.mma.cta_group::2; head
// dim 128, group sizes 4 and 8) four.  S_t = Q_t K_j^T (both operands K-major, 128-byte
// swizzled smem); the softmax threads read their row of S_t with tcgen05.ld,
// compute p = 2^(s*c - m*c) in fp32, write P as bf16 over the first 64 columns
// of S_t, rescale O_t when the running max grew, and signal; O_t += P_t V_j
// reads P from TMEM and V (MN-major) from smem.  S_t(j+1) is issued right
// behind PV_t(j) by the same thread, so it overwrites P_t only after PV_t(j)
// has read it.
//
// K and V come straight out of the cache through one 3-D tensor map per
// sequence, (D, P_b + L_b, Hkv), so rows at or past the sequence's length read
// as zero; the causal mask (keys after the row's position) on the last one or
// two key tiles of a block removes them from the softmax, and an attention
// window adds a lower band (keys before position + 1 - W) and starts the
// block at its window's first tile.
// Every mbarrier wait is bounded (qa_device.cuh): a stuck pipeline records a
// timeout in the error word and the CTA still frees its TMEM and exits.
#include <algorithm>
#include <atomic>

#include "k2_items.h"
#include "qa_device.cuh"

namespace qa {

// max(a, b, c) in one instruction (NaN inputs are ignored, as by fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float k2_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The softmax rescales O only when a row's max grows by more than this many
// powers of two (in the exp2 domain).
constexpr float kRescaleLog2 = 8.f;


// ==================================================================== the kernel
// One CTA per SM walks a fixed share of the work items.  An item is one
// 128-row query block of one sequence for the query heads hpi*pair ..
// hpi*pair + hpi - 1 of a kv head, hpi (heads per item) being 2 unless the
// group size is 1 or two-head items would not give every SM one (a short
// prompt or chunk), then 1: the item's head tiles share every K/V tile of the
// ring.  Items are listed heaviest first
// (most key tiles) and dealt out in snake order (round k gives CTA c item
// k*G + c for even k and k*G + G-1-c for odd k, G = CTAs), which balances the
// key tiles per CTA.  Across items the pipeline never drains:
//   - the TMA warp loads the next item's Q tiles as soon as the current
//     item's last S MMAs have completed (bar_qfree), then its K/V tiles;
//   - the MMA warp issues the next item's first S right behind the current
//     item's last P.V (in issue order, so it overwrites P only after that
//     P.V has read it);
//   - the softmax threads write the item's output (O read from TMEM,
//     normalised, stored) and go on with the next item's first S, which the
//     tensor pipe has already computed.  The next item's first P.V (which
//     overwrites O) is issued only after those threads signal P, i.e. after
//     they have read O.
// Warp roles (320 threads): warps 0-3 softmax of tile 0, warps 4-7 softmax of
// tile 1, warp 8 TMA producer, warp 9 tcgen05 issuer and TMEM owner.
// Tensor memory (512 columns): [0,128) S0/P0, [128,256) S1/P1, [256,256+D) O0,
// [256+D,256+2D) O1.
template <int D>
struct K2PLayout {
    static constexpr int kBoxBytes = 128 * 128;            // 128 rows x 64 bf16
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = kBoxes * kBoxBytes;  // 128 rows x D
    static constexpr int kStages = (D == 128) ? 4 : 8;     // K/V ring
    static constexpr int kQBytes = 2 * kTileBytes;
    static constexpr int kSmemBytes = kQBytes + kStages * kTileBytes + 1024;  // + alignment slack
    static constexpr uint32_t kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kThreads = 320;
    static constexpr int kTmaWarp = 8, kMmaWarp = 9;
};

// The k-th item of this CTA in the snake order (false once its share is done;
// k never below the walk's last call); with shift 1 the two CTAs of a cluster
// take the same items (one per cluster).
template <bool kWindow>
__device__ __forceinline__ bool k2p_item(const K2Params &p, int k, K2Walk &w, K2Item &it,
                                         int shift = 0) {
    return k2_item_at<kWindow>(p, k2_snake_index(k, gridDim.x >> shift, blockIdx.x >> shift), w, it);
}

template <int D, bool kWindow>
__global__ void __launch_bounds__(K2PLayout<D>::kThreads, 1)
    k2p_prefill_kernel(const __grid_constant__ K2Params p) {
    using Lay = K2PLayout<D>;
    constexpr int NS = Lay::kStages;
    const unsigned FULL = 0xffffffffu;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_q, bar_qfree, bar_kv_full[NS], bar_kv_empty[NS];
    __shared__ __align__(8) uint64_t bar_s[2], bar_p[2], bar_pv[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sKV = sQ + Lay::kQBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = p.hpi;  // query heads per item (the same for every item)

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar_q), 1);
        mbar_init(smem_u32(&bar_qfree), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&bar_kv_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bar_s[t]), 1);
            mbar_init(smem_u32(&bar_p[t]), 128);
            mbar_init(smem_u32(&bar_pv[t]), 1);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == Lay::kMmaWarp) {
        tmem_alloc(smem_u32(&s_tmem), Lay::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    griddep_wait();  // as in the CTA-pair form: global data only after this

    if (warp == Lay::kTmaWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&p.tm_q);
            // Test hook: CTA 0 withholds the copy of its first item's V tile 0.
            const uint32_t withheld = (p.fault && blockIdx.x == 0) ? 1u : 0xffffffffu;
            uint32_t g = 0;  // K/V copies requested (K and V of each key tile, in order)
            int nq = 0;      // items whose Q tiles were requested
            bool ok = true;
            K2Walk walk;
            K2Item it;
            for (int k = 0; ok && k2p_item<kWindow>(p, k, walk, it); ++k) {
                // The Q buffers are free once the previous item's last S MMAs are done.
                if (nq > 0 && !mbar_wait(smem_u32(&bar_qfree), (nq - 1) & 1, &s_abort, p.err,
                                         kKernK2, 20, p.wait_ns))
                    break;
                prefetch_tmap(&p.tm_k[it.b]);
                prefetch_tmap(&p.tm_v[it.b]);
                const uint32_t bq = smem_u32(&bar_q);
                mbar_expect_tx(bq, ntiles * Lay::kTileBytes);
                for (int t = 0; t < ntiles; ++t)
                    for (int x = 0; x < Lay::kBoxes; ++x)
                        tma_load_3d(sQ + t * Lay::kTileBytes + x * Lay::kBoxBytes, &p.tm_q, x * 64,
                                    it.h0 + t, it.row0, bq);
                ++nq;
                for (int idx = 0; idx < 2 * it.nkv; ++idx, ++g) {
                    const int st = g % NS;
                    if (g >= NS && !mbar_wait(smem_u32(&bar_kv_empty[st]), ((g / NS) - 1) & 1,
                                              &s_abort, p.err, kKernK2, 21, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (g == withheld) continue;
                    const uint32_t fb = smem_u32(&bar_kv_full[st]);
                    mbar_expect_tx(fb, Lay::kTileBytes);
                    const uint32_t dst = sKV + st * Lay::kTileBytes;
                    const int key0 = (it.j0 + (idx >> 1)) * 128;
                    for (int x = 0; x < Lay::kBoxes; ++x) {
                        if (idx & 1) {
                            tma_load_3d(dst + x * Lay::kBoxBytes, &p.tm_v[it.b], x * 64, key0, it.kvh, fb);
                        } else {  // two 64-row boxes stack into the same swizzled layout
                            for (int h = 0; h < 2; ++h)
                                tma_load_3d(dst + x * Lay::kBoxBytes + h * (Lay::kBoxBytes / 2),
                                            &p.tm_k[it.b], x * 64, key0 + 64 * h, it.kvh, fb);
                        }
                    }
                }
            }
            // Never leave a copy in flight: bounded waits for the last ones and Q.
            int dummy = 0;
            for (uint32_t i = g > NS ? g - NS : 0; i < g; ++i)
                if (i != withheld)
                    mbar_wait(smem_u32(&bar_kv_full[i % NS]), (i / NS) & 1, &dummy, p.err, kKernK2,
                              22, p.wait_ns);
            if (nq > 0)
                mbar_wait(smem_u32(&bar_q), (nq - 1) & 1, &dummy, p.err, kKernK2, 23, p.wait_ns);
        }
    } else if (warp == Lay::kMmaWarp) {
        // ------------------------------------------------------------ tcgen05 issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
            const uint32_t tS[2] = {tmem, tmem + Lay::kColS1};
            const uint32_t tO[2] = {tmem + Lay::kColO0, tmem + Lay::kColO1};
            // Descriptors are built once per operand tile; a K-step only moves the
            // start address (bits 0-13, 16-byte units, never carrying out at
            // shared-memory addresses): one 32-bit add on the low word.
            auto desc_at = [](uint64_t base, uint32_t byte_off) -> uint64_t {
                return (base & 0xFFFFFFFF00000000ull) |
                       static_cast<uint32_t>(static_cast<uint32_t>(base) + (byte_off >> 4));
            };
            const uint64_t dQ[2] = {sdesc_sw128(sQ, 16, 1024),
                                    sdesc_sw128(sQ + Lay::kTileBytes, 16, 1024)};
            // S_t = Q_t K^T: K-major operands, 128-byte swizzle, 8-row groups 1024 B
            // apart; K-step k of 16 elements = 32 bytes inside the 128-byte row of box k/4.
            auto issue_s = [&](int t, int st) {
                const uint64_t dK = sdesc_sw128(sKV + st * Lay::kTileBytes, 16, 1024);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k / 4) * Lay::kBoxBytes + (k % 4) * 32;
                    mma_ss(tS[t], desc_at(dQ[t], off), desc_at(dK, off), idesc_qk, k > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t V: P (bf16, 2 per column) from TMEM; V MN-major in smem, 64-wide
            // d blocks one box apart, 8-row key groups 1024 B apart; a K-step of 16
            // keys = 2048 bytes.
            auto issue_pv = [&](int t, int st, bool acc) {
                const uint64_t dV = sdesc_sw128(sKV + st * Lay::kTileBytes, Lay::kBoxBytes, 1024);
#pragma unroll
                for (int k = 0; k < 128 / 16; ++k)
                    mma_ts(tO[t], tS[t] + k * 8, desc_at(dV, k * 2048), idesc_pv,
                           (acc || k > 0) ? 1u : 0u);
            };
            uint32_t g = 0;          // K/V copies consumed, in the producer's order
            uint32_t iter = 0;       // key-tile iterations (phases of bar_s / bar_p)
            uint32_t committed = 0;  // ring slots handed back (one per copy, in order)
            int nq = 0, nqfree = 0;
            bool ok = true;
            K2Walk walk;
            K2Item it;
            for (int k = 0; ok && k2p_item<kWindow>(p, k, walk, it); ++k) {
                ok = mbar_wait(smem_u32(&bar_q), nq & 1, &s_abort, p.err, kKernK2, 24, p.wait_ns);
                ++nq;
                if (ok)
                    ok = mbar_wait(smem_u32(&bar_kv_full[g % NS]), (g / NS) & 1, &s_abort, p.err,
                                   kKernK2, 25, p.wait_ns);
                if (!ok) break;
                tc_fence_after();
                // The first S of the item: the previous item's last P.V were issued
                // before, so they have read the P columns these overwrite.
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (t < ntiles) {
                        issue_s(t, g % NS);
                        mma_commit(smem_u32(&bar_s[t]));
                    }
                }
                if (it.nkv == 1) {
                    mma_commit(smem_u32(&bar_qfree));
                    ++nqfree;
                }
                mma_commit(smem_u32(&bar_kv_empty[g % NS]));
                ++committed;
                for (int j = 0; ok && j < it.nkv; ++j) {
                    const uint32_t iv = g + 2 * j + 1, ik = g + 2 * j + 2;
                    const int sv = iv % NS, sk = ik % NS;
                    const bool more = j + 1 < it.nkv;
                    ok = mbar_wait(smem_u32(&bar_kv_full[sv]), (iv / NS) & 1, &s_abort, p.err,
                                   kKernK2, 26, p.wait_ns);
                    if (ok && more)
                        ok = mbar_wait(smem_u32(&bar_kv_full[sk]), (ik / NS) & 1, &s_abort, p.err,
                                       kKernK2, 27, p.wait_ns);
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (!ok || t >= ntiles) break;
                        ok = mbar_wait(smem_u32(&bar_p[t]), iter & 1, &s_abort, p.err, kKernK2, 28,
                                       p.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(t, sv, j > 0);
                        if (!more) mma_commit(smem_u32(&bar_pv[t]));  // O_t of the item is final
                        if (t == ntiles - 1) {
                            mma_commit(smem_u32(&bar_kv_empty[sv]));
                            ++committed;
                        }
                        if (more) {
                            issue_s(t, sk);
                            mma_commit(smem_u32(&bar_s[t]));
                            if (t == ntiles - 1) {
                                mma_commit(smem_u32(&bar_kv_empty[sk]));
                                ++committed;
                            }
                        }
                    }
                    if (ok && more && j + 2 == it.nkv) {  // the S just issued are the item's last
                        mma_commit(smem_u32(&bar_qfree));
                        ++nqfree;
                    }
                    ++iter;
                }
                g += 2 * it.nkv;
            }
            // Drain: every commit above must have arrived before the CTA exits.
            int dummy = 0;
            for (uint32_t i = committed > NS ? committed - NS : 0; i < committed; ++i)
                mbar_wait(smem_u32(&bar_kv_empty[i % NS]), (i / NS) & 1, &dummy, p.err, kKernK2,
                          29, p.wait_ns);
            if (nqfree > 0)
                mbar_wait(smem_u32(&bar_qfree), (nqfree - 1) & 1, &dummy, p.err, kKernK2, 30,
                          p.wait_ns);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = warp >> 2;  // 0 or 1
        if (t < ntiles) {
            const int r = (warp & 3) * 32 + lane;  // row of the tile == TMEM lane
            const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const uint32_t tS = tmem + (t ? Lay::kColS1 : 0u) + lane_off;
            const uint32_t tO = tmem + (t ? Lay::kColO1 : Lay::kColO0) + lane_off;
            const float c = p.scale_log2;
            uint32_t iter = 0;
            int nitem = 0;
            bool ok = true;
            K2Walk walk;
            K2Item it;
            for (int k = 0; ok && k2p_item<kWindow>(p, k, walk, it); ++k) {
                const int qpos = it.qmin + r;  // this row's position
                // mref: the row's reference max (raw scores); it moves only when the
                // row max exceeds it by more than kRescaleLog2 / c, so O is rescaled
                // rarely; p = 2^(s*c - mref*c) stays below 2^kRescaleLog2, and
                // out = O / l is exact for any mref.
                float mref = -INFINITY, l = 0.f;
                for (int j = 0; j < it.nkv; ++j, ++iter) {
                    ok = mbar_wait(smem_u32(&bar_s[t]), iter & 1, &s_abort, p.err, kKernK2, 31,
                                   p.wait_ns);
                    ok = __all_sync(FULL, ok);
                    if (!ok) break;
                    tc_fence_after();
                    const int jt = it.j0 + j;         // key tile
                    const int thr = qpos - jt * 128;  // last visible key index in the tile
                    const int tlo = kWindow ? qpos + 1 - p.window - jt * 128 : 0;
                    uint32_t sr[128];
                    {
                        uint32_t(&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr);
                        uint32_t(&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 32);
                        uint32_t(&s2)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 64);
                        uint32_t(&s3)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 96);
                        tmem_ld32_async(tS, s0);
                        tmem_ld32_async(tS + 32, s1);
                        tmem_ld32_async(tS + 64, s2);
                        tmem_ld32_async(tS + 96, s3);
                        tmem_wait_ld4(s0, s1, s2, s3);
                    }
                    if (jt >= it.jmask || tlo > 0) {
#pragma unroll
                        for (int i = 0; i < 128; ++i)
                            if (i > thr || i < tlo) sr[i] = __float_as_uint(-INFINITY);
                    }
                    float mx8[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        mx8[q] = fmaxf(__uint_as_float(sr[q]), __uint_as_float(sr[8 + q]));
#pragma unroll
                    for (int i = 16; i < 128; i += 16) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            mx8[q] = fmax3(mx8[q], __uint_as_float(sr[i + q]),
                                           __uint_as_float(sr[i + 8 + q]));
                    }
                    const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                                           fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                    bool rescale = false;
                    float alpha = 1.f;
                    if (j == 0) {
                        mref = mx == -INFINITY ? 0.f : mx;  // a window can mask a whole tile
                    } else {
                        const bool grow = (mx - mref) * c > kRescaleLog2;
                        rescale = __any_sync(FULL, grow);
                        if (grow) {
                            alpha = k2_ex2((mref - mx) * c);
                            mref = mx;
                            l *= alpha;
                        }
                    }
                    const float2 c2 = make_float2(c, c);
                    const float2 n2 = make_float2(-mref * c, -mref * c);
                    float2 sum4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) sum4[q] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int col = ch * 32 + 2 * i;
                            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[col]),
                                                                    __uint_as_float(sr[col + 1])),
                                                        c2, n2);
                            const float2 pv = make_float2(k2_ex2(x.x), k2_ex2(x.y));
                            pk[i] = pack_bf16(pv.x, pv.y);
                            sum4[i & 3] = __fadd2_rn(sum4[i & 3], pv);
                        }
                        tmem_st16(tS + ch * 16, pk);
                    }
                    const float2 sp =
                        __fadd2_rn(__fadd2_rn(sum4[0], sum4[1]), __fadd2_rn(sum4[2], sum4[3]));
                    l += sp.x + sp.y;
                    if (rescale) {
                        // P.V_t(j-1) is complete: the commit that signalled S_t(j)
                        // tracks every tcgen05 operation issued before it.
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int ch = 0; ch < D / 32; ++ch) {
                            uint32_t u[32];
                            tmem_ld32(tO + ch * 32, u);
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float2 v = __fmul2_rn(make_float2(__uint_as_float(u[2 * i]),
                                                                        __uint_as_float(u[2 * i + 1])),
                                                            a2);
                                u[2 * i] = __float_as_uint(v.x);
                                u[2 * i + 1] = __float_as_uint(v.y);
                            }
                            tmem_st32(tO + ch * 32, u);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bar_p[t]));
                }
                if (!ok) break;
                // The item's output: O_t / l in bf16.  The next item's first P.V,
                // which overwrites O_t, waits for this warpgroup's next signal.
                ok = mbar_wait(smem_u32(&bar_pv[t]), nitem & 1, &s_abort, p.err, kKernK2, 32,
                               p.wait_ns);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                ++nitem;
                tc_fence_after();
                const float inv = 1.f / l;
                const int row = it.qb * 128 + r;  // new token index within the sequence
                const bool valid = row < it.L;
                __nv_bfloat16 *dst =
                    p.out + (static_cast<int64_t>(p.cu[it.b] + row) * p.Hq + it.h0 + t) * D;
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t u[32];
                    tmem_ld32(tO + ch * 32, u);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16(__uint_as_float(u[2 * i]) * inv,
                                         __uint_as_float(u[2 * i + 1]) * inv);
                    if (valid) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == Lay::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

// ==================================================================== the CTA-pair form
// Two CTAs of a cluster (two SMs) share every item: one 128-row query block of
// a sequence for four query heads h0 .. h0 + 3 of a kv head; CTA r holds heads
// h0 + 2r and h0 + 2r + 1 as its two tiles (same rows, same causal mask, same
// key tiles).  One thread of CTA 0 issues every tensor-core operation of both
// as tcgen05.mma.cta_group::2 with M = 256 (CTA 0's tile rows, then CTA 1's):
//   - S_t = Q_t K_j^T reads each CTA's own Q tile and half of the key tile from
//     each CTA (keys 0-63 from CTA 0, 64-127 from CTA 1): 6 KB of shared memory
//     per SM and 128x128x16 step, against 8 KB when one CTA holds both operands;
//   - O_t += P_t V_j reads P from each CTA's tensor memory and half of V's
//     columns from each (d 0-63 from CTA 0, 64-127 from CTA 1).
// So each SM loads half of every K/V tile.  Each CTA's TMA warp copies its own
// Q tiles and halves, completing on CTA 0's barriers (CTA 0 arms them with the
// bytes of both); every commit is multicast to both CTAs; each softmax warp of
// either CTA signals CTA 0 once per key tile.  Both TMA warps run the same
// schedule against the same (multicast) barrier phases and their waits ignore
// the abort flag, so they issue the same copies: CTA 0's final waits cover
// CTA 1's copies, and a closing cluster barrier keeps either CTA resident
// until the other no longer touches it.  Tensor memory as in the one-CTA form.
struct K2CLayout {
    static constexpr int D = 128;
    static constexpr int kQBoxBytes = 128 * 128;         // 128 rows x 64 bf16
    static constexpr int kQTileBytes = 2 * kQBoxBytes;   // 128 rows x D
    static constexpr int kQBytes = 2 * kQTileBytes;      // this CTA's two tiles of one item
    static constexpr int kQSlots = 2;                    // item k's Q in slot k mod kQSlots
    static constexpr int kKBoxBytes = 64 * 128;          // 64 keys x 64 bf16
    static constexpr int kHalfBytes = 2 * kKBoxBytes;    // this CTA's half of a K or V tile
    static constexpr int kStages = 4;                    // ring of halves: 2 key tiles
    static constexpr int kStageOutBytes = 32 * 128;      // per softmax warp: 32 rows x 64 bf16
    static constexpr int kSmemBytes =
        kQSlots * kQBytes + kStages * kHalfBytes + 8 * kStageOutBytes + 1024;
    static constexpr uint32_t kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kThreads = 352;
    static constexpr int kTmaWarp = 8, kMmaWarp = 9, kQWarp = 10;
};

template <bool kWindow>
__global__ void __launch_bounds__(K2CLayout::kThreads, 1)
    k2c_prefill_kernel(const __grid_constant__ K2Params p) {
    using Lay = K2CLayout;
    constexpr int NS = Lay::kStages;
    constexpr int D = Lay::D;
    constexpr uint16_t kBoth = 0x3;  // commit multicast: both CTAs of the pair
    const unsigned FULL = 0xffffffffu;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_q[2], bar_qfree[2], bar_kv_full[NS], bar_kv_empty[NS];
    __shared__ __align__(8) uint64_t bar_s[2], bar_p[2], bar_pv[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sQ = smem_u32(smem);  // item k's Q tiles in slot k mod 2
    const uint32_t sKV = sQ + Lay::kQSlots * Lay::kQBytes;
    uint8_t *sOut = smem + Lay::kQSlots * Lay::kQBytes + NS * Lay::kHalfBytes;  // output staging
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs of the pair
    const int pair_id = blockIdx.x >> 1;

    if (threadIdx.x == 0) {
        // Used in CTA 0 only: bar_q, bar_kv_full (both CTAs' bytes), bar_p (the
        // four softmax warps of each CTA per tile).  In both: the rest.
        for (int q = 0; q < 2; ++q) {
            mbar_init(smem_u32(&bar_q[q]), 1);
            mbar_init(smem_u32(&bar_qfree[q]), 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&bar_kv_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bar_s[t]), 1);
            mbar_init(smem_u32(&bar_p[t]), 8);
            mbar_init(smem_u32(&bar_pv[t]), 1);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == Lay::kMmaWarp) {
        tmem_alloc_pair(smem_u32(&s_tmem), Lay::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised, tensor memory allocated
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // Launched as a programmatic dependent: the set-up above may overlap the
    // previous kernel's end (the norm/RoPE/append kernel, which signals at
    // its start); every read and write of global data comes after this wait.
    griddep_wait();

    if (warp == Lay::kTmaWarp) {
        // ------------------------------------------------------------ K/V producer (both CTAs)
        int no_abort = 0;  // see above: the producers' waits do not follow s_abort
        if (lane == 0) {
            // Test hook: both CTAs of the first pair withhold their halves of its
            // first item's V tile 0 (no byte of that copy is ever in flight).
            const uint32_t withheld = (p.fault && pair_id == 0) ? 1u : 0xffffffffu;
            uint32_t g = 0;
            bool ok = true;
            K2Walk walk;
            K2Item it;
            for (int k = 0; ok && k2p_item<kWindow>(p, k, walk, it, 1); ++k) {
                prefetch_tmap(&p.tm_k[it.b]);
                prefetch_tmap(&p.tm_v[it.b]);
                for (int idx = 0; idx < 2 * it.nkv; ++idx, ++g) {
                    const int st = g % NS;
                    if (g >= NS && !mbar_wait(smem_u32(&bar_kv_empty[st]), ((g / NS) - 1) & 1,
                                              &no_abort, p.err, kKernK2, 41, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (g == withheld) continue;
                    const uint32_t fb = smem_u32(&bar_kv_full[st]);
                    if (rank == 0) mbar_expect_tx(fb, 2 * Lay::kHalfBytes);
                    const uint32_t fb_lead = map_rank(fb, 0);
                    const uint32_t dst = sKV + st * Lay::kHalfBytes;
                    const int key0 = (it.j0 + (idx >> 1)) * 128;
                    if (idx & 1) {  // V: columns 64r .. 64r + 63 of 128 keys
                        tma_load_3d_pair(dst, &p.tm_v[it.b], 64 * static_cast<int>(rank), key0,
                                         it.kvh, fb_lead);
                    } else {        // K: keys 64r .. 64r + 63 of the tile, all D columns
                        for (int x = 0; x < 2; ++x)
                            tma_load_3d_pair(dst + x * Lay::kKBoxBytes, &p.tm_k[it.b], x * 64,
                                             key0 + 64 * static_cast<int>(rank), it.kvh, fb_lead);
                    }
                }
            }
            if (rank == 0) {
                // Never leave a copy in flight: both CTAs' last copies complete on
                // these barriers (bounded waits).
                int dummy = 0;
                for (uint32_t i = g > NS ? g - NS : 0; i < g; ++i)
                    if (i != withheld)
                        mbar_wait(smem_u32(&bar_kv_full[i % NS]), (i / NS) & 1, &dummy, p.err,
                                  kKernK2, 42, p.wait_ns);
            }
        }
    } else if (warp == Lay::kQWarp) {
        // ------------------------------------------------------------ Q producer (both CTAs)
        // A warp of its own, so its waits never hold up the K/V copies: each
        // item's Q tiles load as soon as their slot is free, about an item ahead.
        int no_abort = 0;
        constexpr int QS = Lay::kQSlots;
        if (lane == 0) {
            prefetch_tmap(&p.tm_q);
            int nq = 0;
            K2Walk walk;
            K2Item it;
            for (int k = 0; k2p_item<kWindow>(p, k, walk, it, 1); ++k) {
                // Q slot k mod kQSlots is free once the last S MMAs of the item
                // before that used it are done.
                const int qs = k % QS;
                if (k >= QS && !mbar_wait(smem_u32(&bar_qfree[qs]), ((k / QS) - 1) & 1, &no_abort,
                                          p.err, kKernK2, 40, p.wait_ns))
                    break;
                const uint32_t bq = smem_u32(&bar_q[qs]);
                if (rank == 0) mbar_expect_tx(bq, 2 * Lay::kQBytes);
                const uint32_t bq_lead = map_rank(bq, 0);
                for (int t = 0; t < 2; ++t)
                    for (int x = 0; x < 2; ++x)
                        tma_load_3d_pair(sQ + qs * Lay::kQBytes + t * Lay::kQTileBytes +
                                             x * Lay::kQBoxBytes,
                                         &p.tm_q, x * 64, it.h0 + 2 * static_cast<int>(rank) + t,
                                         it.row0, bq_lead);
                ++nq;
                // The next item's Q tiles into L2 meanwhile: a short item leaves
                // less time than a copy from HBM takes.
                K2Item nx;
                if (k2p_item<kWindow>(p, k + 1, walk, nx, 1))
                    for (int t = 0; t < 2; ++t)
                        for (int x = 0; x < 2; ++x)
                            tma_prefetch_3d(&p.tm_q, x * 64, nx.h0 + 2 * static_cast<int>(rank) + t,
                                            nx.row0);
            }
            if (rank == 0) {
                int dummy = 0;
                for (int i = nq > QS ? nq - QS : 0; i < nq; ++i)
                    mbar_wait(smem_u32(&bar_q[i % QS]), (i / QS) & 1, &dummy, p.err, kKernK2, 43,
                              p.wait_ns);
            }
        }
    } else if (warp == Lay::kMmaWarp) {
        // ------------------------------------------------------------ tcgen05 issuer (CTA 0)
        if (rank == 0 && lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(256, 128, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(256, D, false, true);
            const uint32_t tS[2] = {tmem, tmem + Lay::kColS1};
            const uint32_t tO[2] = {tmem + Lay::kColO0, tmem + Lay::kColO1};
            auto desc_at = [](uint64_t base, uint32_t byte_off) -> uint64_t {
                return (base & 0xFFFFFFFF00000000ull) |
                       static_cast<uint32_t>(static_cast<uint32_t>(base) + (byte_off >> 4));
            };
            uint64_t dQ[2];  // the current item's Q tiles
            // S_t = Q_t K^T: K-major, 128-byte swizzle, 8-row groups 1024 B apart;
            // K-step k (16 columns = 32 bytes) inside box k/4 of each operand.
            auto issue_s = [&](int t, int st) {
                const uint64_t dK = sdesc_sw128(sKV + st * Lay::kHalfBytes, 16, 1024);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss_pair(tS[t], desc_at(dQ[t], (k / 4) * Lay::kQBoxBytes + (k % 4) * 32),
                                desc_at(dK, (k / 4) * Lay::kKBoxBytes + (k % 4) * 32), idesc_qk,
                                k > 0 ? 1u : 0u);
            };
            // O_t += P_t V: P from tensor memory; this CTA's 64 columns of V
            // MN-major (one 128-byte swizzle atom wide), 8-key groups 1024 B
            // apart; a K-step of 16 keys = 2048 bytes.
            auto issue_pv = [&](int t, int st, bool acc) {
                const uint64_t dV = sdesc_sw128(sKV + st * Lay::kHalfBytes, Lay::kHalfBytes, 1024);
#pragma unroll
                for (int k = 0; k < 128 / 16; ++k)
                    mma_ts_pair(tO[t], tS[t] + k * 8, desc_at(dV, k * 2048), idesc_pv,
                                (acc || k > 0) ? 1u : 0u);
            };
            uint32_t g = 0, iter = 0, committed = 0;
            int nq = 0, nqfree = 0;
            bool ok = true;
            K2Walk walk;
            K2Item it;
            for (int k = 0; ok && k2p_item<kWindow>(p, k, walk, it, 1); ++k) {
                const int qs = k % Lay::kQSlots;
                ok = mbar_wait(smem_u32(&bar_q[qs]), (k / Lay::kQSlots) & 1, &s_abort, p.err, kKernK2, 44,
                               p.wait_ns);
                dQ[0] = sdesc_sw128(sQ + qs * Lay::kQBytes, 16, 1024);
                dQ[1] = sdesc_sw128(sQ + qs * Lay::kQBytes + Lay::kQTileBytes, 16, 1024);
                ++nq;
                if (ok)
                    ok = mbar_wait(smem_u32(&bar_kv_full[g % NS]), (g / NS) & 1, &s_abort, p.err,
                                   kKernK2, 45, p.wait_ns);
                if (!ok) break;
                tc_fence_after();
                for (int t = 0; t < 2; ++t) {
                    issue_s(t, g % NS);
                    mma_commit_pair(smem_u32(&bar_s[t]), kBoth);
                }
                if (it.nkv == 1) {
                    mma_commit_pair(smem_u32(&bar_qfree[qs]), kBoth);
                    ++nqfree;
                }
                mma_commit_pair(smem_u32(&bar_kv_empty[g % NS]), kBoth);
                ++committed;
                for (int j = 0; ok && j < it.nkv; ++j) {
                    const uint32_t iv = g + 2 * j + 1, ik = g + 2 * j + 2;
                    const int sv = iv % NS, sk = ik % NS;
                    const bool more = j + 1 < it.nkv;
                    ok = mbar_wait(smem_u32(&bar_kv_full[sv]), (iv / NS) & 1, &s_abort, p.err,
                                   kKernK2, 46, p.wait_ns);
                    if (ok && more)
                        ok = mbar_wait(smem_u32(&bar_kv_full[sk]), (ik / NS) & 1, &s_abort, p.err,
                                       kKernK2, 47, p.wait_ns);
                    for (int t = 0; ok && t < 2; ++t) {
                        // P_t of both CTAs (four warps each)
                        ok = mbar_wait(smem_u32(&bar_p[t]), iter & 1, &s_abort, p.err, kKernK2, 48,
                                       p.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(t, sv, j > 0);
                        if (!more) mma_commit_pair(smem_u32(&bar_pv[t]), kBoth);  // O_t of the item is final
                        if (t == 1) {
                            mma_commit_pair(smem_u32(&bar_kv_empty[sv]), kBoth);
                            ++committed;
                        }
                        if (more) {
                            issue_s(t, sk);
                            mma_commit_pair(smem_u32(&bar_s[t]), kBoth);
                            if (t == 1) {
                                mma_commit_pair(smem_u32(&bar_kv_empty[sk]), kBoth);
                                ++committed;
                            }
                        }
                    }
                    if (ok && more && j + 2 == it.nkv) {
                        mma_commit_pair(smem_u32(&bar_qfree[qs]), kBoth);
                        ++nqfree;
                    }
                    ++iter;
                }
                g += 2 * it.nkv;
            }
            // Drain: every tensor-core operation on either CTA is done before
            // the closing barrier (a commit tracks every earlier operation).
            int dummy = 0;
            for (uint32_t i = committed > NS ? committed - NS : 0; i < committed; ++i)
                mbar_wait(smem_u32(&bar_kv_empty[i % NS]), (i / NS) & 1, &dummy, p.err, kKernK2,
                          49, p.wait_ns);
            for (int i = nqfree > Lay::kQSlots ? nqfree - Lay::kQSlots : 0; i < nqfree; ++i)
                mbar_wait(smem_u32(&bar_qfree[i % Lay::kQSlots]), (i / Lay::kQSlots) & 1, &dummy, p.err,
                          kKernK2, 50,
                          p.wait_ns);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups (both CTAs)
        const int t = warp >> 2;                 // tile 0 or 1
        const int r = (warp & 3) * 32 + lane;    // row of the tile == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + (t ? Lay::kColS1 : 0u) + lane_off;
        const uint32_t tO = tmem + (t ? Lay::kColO1 : Lay::kColO0) + lane_off;
        const uint32_t bp_lead = map_rank(smem_u32(&bar_p[t]), 0);
        const float c = p.scale_log2;
        uint32_t iter = 0;
        bool ok = true;
        int nitem = 0;
        K2Walk walk;
        K2Item it;
        for (int k = 0; ok && k2p_item<kWindow>(p, k, walk, it, 1); ++k) {
            const int qpos = it.qmin + r;
            float mref = -INFINITY, l = 0.f;  // as in the one-CTA form
            for (int j = 0; j < it.nkv; ++j, ++iter) {
                ok = mbar_wait(smem_u32(&bar_s[t]), iter & 1, &s_abort, p.err, kKernK2, 51,
                               p.wait_ns);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc_fence_after();
                const int jt = it.j0 + j;
                const int thr = qpos - jt * 128;
                const int tlo = kWindow ? qpos + 1 - p.window - jt * 128 : 0;
                uint32_t sr[128];
                {
                    uint32_t(&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr);
                    uint32_t(&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 32);
                    uint32_t(&s2)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 64);
                    uint32_t(&s3)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 96);
                    tmem_ld32_async(tS, s0);
                    tmem_ld32_async(tS + 32, s1);
                    tmem_ld32_async(tS + 64, s2);
                    tmem_ld32_async(tS + 96, s3);
                    tmem_wait_ld4(s0, s1, s2, s3);
                }
                if (jt >= it.jmask || tlo > 0) {
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i > thr || i < tlo) sr[i] = __float_as_uint(-INFINITY);
                }
                float mx8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    mx8[q] = fmaxf(__uint_as_float(sr[q]), __uint_as_float(sr[8 + q]));
#pragma unroll
                for (int i = 16; i < 128; i += 16) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        mx8[q] = fmax3(mx8[q], __uint_as_float(sr[i + q]), __uint_as_float(sr[i + 8 + q]));
                }
                const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                                       fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                bool rescale = false;
                float alpha = 1.f;
                if (j == 0) {
                    mref = mx == -INFINITY ? 0.f : mx;
                } else {
                    const bool grow = (mx - mref) * c > kRescaleLog2;
                    rescale = __any_sync(FULL, grow);
                    if (grow) {
                        alpha = k2_ex2((mref - mx) * c);
                        mref = mx;
                        l *= alpha;
                    }
                }
                const float2 c2 = make_float2(c, c);
                const float2 n2 = make_float2(-mref * c, -mref * c);
                float2 sum4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) sum4[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int col = ch * 32 + 2 * i;
                        const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[col]),
                                                                __uint_as_float(sr[col + 1])),
                                                    c2, n2);
                        const float2 pv = make_float2(k2_ex2(x.x), k2_ex2(x.y));
                        pk[i] = pack_bf16(pv.x, pv.y);
                        sum4[i & 3] = __fadd2_rn(sum4[i & 3], pv);
                    }
                    tmem_st16(tS + ch * 16, pk);
                }
                const float2 sp = __fadd2_rn(__fadd2_rn(sum4[0], sum4[1]), __fadd2_rn(sum4[2], sum4[3]));
                l += sp.x + sp.y;
                if (rescale) {
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t u[32];
                        tmem_ld32(tO + ch * 32, u);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 v = __fmul2_rn(make_float2(__uint_as_float(u[2 * i]),
                                                                    __uint_as_float(u[2 * i + 1])),
                                                        a2);
                            u[2 * i] = __float_as_uint(v.x);
                            u[2 * i + 1] = __float_as_uint(v.y);
                        }
                        tmem_st32(tO + ch * 32, u);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(bp_lead);  // this warp's 32 rows of P_t
            }
            if (!ok) break;
            ok = mbar_wait(smem_u32(&bar_pv[t]), nitem & 1, &s_abort, p.err, kKernK2, 52, p.wait_ns);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            ++nitem;
            tc_fence_after();
            // O_t / l in bf16 through this warp's staging area, half a row (64
            // columns, 128 bytes) at a time: each lane writes its own row (16-byte
            // chunks XOR-swizzled by row, so the 32 rows spread over all banks),
            // then the warp reads back four rows x 128 bytes per instruction and
            // stores whole 128-byte lines (rows past the sequence's end skipped).
            const float inv = 1.f / l;
            uint8_t *stg = sOut + warp * Lay::kStageOutBytes;
            const int rw = lane >> 3, cw = lane & 7;  // read-back: row within a group of 4, chunk
            const int row_base = it.qb * 128 + (warp & 3) * 32;  // token index of the warp's row 0
            __nv_bfloat16 *obase = p.out + (static_cast<int64_t>(p.cu[it.b]) * p.Hq + it.h0 +
                                            2 * static_cast<int>(rank) + t) * D;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t u[32];
                    tmem_ld32(tO + h * 64 + c2 * 32, u);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 v = make_uint4(
                            pack_bf16(__uint_as_float(u[8 * i]) * inv, __uint_as_float(u[8 * i + 1]) * inv),
                            pack_bf16(__uint_as_float(u[8 * i + 2]) * inv, __uint_as_float(u[8 * i + 3]) * inv),
                            pack_bf16(__uint_as_float(u[8 * i + 4]) * inv, __uint_as_float(u[8 * i + 5]) * inv),
                            pack_bf16(__uint_as_float(u[8 * i + 6]) * inv, __uint_as_float(u[8 * i + 7]) * inv));
                        const int chunk = c2 * 4 + i;
                        *reinterpret_cast<uint4 *>(stg + lane * 128 + ((chunk ^ (lane & 7)) << 4)) = v;
                    }
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = 4 * i + rw;  // row within the warp's 32
                    const uint4 v =
                        *reinterpret_cast<const uint4 *>(stg + rr * 128 + ((cw ^ (rr & 7)) << 4));
                    if (row_base + rr < it.L)
                        reinterpret_cast<uint4 *>(obase + static_cast<int64_t>(row_base + rr) * p.Hq * D +
                                                  h * 64)[cw] = v;
                }
                __syncwarp();  // read back before the next half overwrites the stage
            }
        }
    }

    tc_fence_before();
    cluster_sync_all();  // neither CTA leaves while the other may still signal or read it
    if (warp == Lay::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, Lay::kTmemCols);
    }
}

// SM count of the current device (cached per device).
static int k2_num_sms() {
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int known = cache[dev].load(std::memory_order_acquire);
        if (known > 0) return known;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev].store(sms, std::memory_order_release);
    return sms;
}

// Clusters of two CTA-pair prefill CTAs that can be resident at once on the
// current device (cached per device; 0 when the device cannot hold one).
template <bool kWindow>
static int k2c_clusters() {
    static std::atomic<int> cache[32] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 32) {
        const int known = cache[dev].load(std::memory_order_acquire);
        if (known != 0) return known > 0 ? known : 0;
    }
    int n = 0;
    bool failed = false;
    if (cudaFuncSetAttribute(k2c_prefill_kernel<kWindow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             K2CLayout::kSmemBytes) != cudaSuccess) {
        failed = true;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(K2CLayout::kThreads);
        cfg.dynamicSmemBytes = K2CLayout::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, k2c_prefill_kernel<kWindow>, &cfg) != cudaSuccess) {
            n = 0;
            failed = true;
        }
    }
    if (failed) cudaGetLastError();  // the failed query's error is not left for the caller
    if (dev < 32) cache[dev].store(n > 0 ? n : -1, std::memory_order_release);
    return n;
}

// The CTA-pair form: items of four query heads, one cluster of two per item
// at a time, as many clusters as can be resident (persistent).
template <bool kWindow>
static cudaError_t launch_k2c(const K2Params &p, int items4, int clusters, cudaStream_t stream) {
    K2Params q = p;
    q.hpi = 4;
    q.npairs = p.G / 4;
    q.nitems = items4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * std::min(items4, clusters), 1, 1);
    cfg.blockDim = dim3(K2CLayout::kThreads);
    cfg.dynamicSmemBytes = K2CLayout::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k2c_prefill_kernel<kWindow>, q);
}

template <int D, bool kWindow>
static cudaError_t launch_k2_t(const K2Params &p, int nitems, cudaStream_t stream) {
    if (D == 128 && p.G % 4 == 0) {
        // Four-head items on CTA pairs whenever every resident pair gets one.
        const int items4 = nitems / p.npairs * (p.G / 4);
        const int clusters = k2c_clusters<kWindow>();
        if (clusters > 0 && items4 >= clusters) return launch_k2c<kWindow>(p, items4, clusters, stream);
    }
    using Lay = K2PLayout<D>;
    constexpr int smem = Lay::kSmemBytes;
    static std::atomic<unsigned> configured{0u};  // devices 0..31 set up (one bit each)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 32 || !((configured.load(std::memory_order_acquire) >> dev) & 1u)) {
        cudaError_t e = cudaFuncSetAttribute(k2p_prefill_kernel<D, kWindow>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev < 32) configured.fetch_or(1u << dev, std::memory_order_release);
    }
    const int sms = k2_num_sms();
    if (sms <= 0) return cudaErrorInvalidDevice;
    K2Params q = p;
    q.hpi = p.G > 1 ? 2 : 1;
    q.npairs = (p.G + q.hpi - 1) / q.hpi;
    q.nitems = nitems / p.npairs * q.npairs;
    if (q.hpi == 2 && q.nitems < sms) {
        // Fewer two-head items than SMs (a short prompt or chunk): one query
        // head per item, twice the work units.
        q.hpi = 1;
        q.npairs = p.G;
        q.nitems = nitems / p.npairs * q.npairs;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(q.nitems, sms), 1, 1);
    cfg.blockDim = dim3(Lay::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k2p_prefill_kernel<D, kWindow>, q);
}

cudaError_t launch_k2(const K2Params &p, int D, int nitems, cudaStream_t stream) {
    if (nitems <= 0) return cudaSuccess;
    const bool win = p.window > 0;
    if (D == 128)
        return win ? launch_k2_t<128, true>(p, nitems, stream) : launch_k2_t<128, false>(p, nitems, stream);
    if (D == 64)
        return win ? launch_k2_t<64, true>(p, nitems, stream) : launch_k2_t<64, false>(p, nitems, stream);
    return cudaErrorInvalidValue;
}

}  // namespace qa
