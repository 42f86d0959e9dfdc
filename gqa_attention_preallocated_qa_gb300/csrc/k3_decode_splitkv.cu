// k3_decode_splitkv.cu -- K3: one fused launch per decode step of one layer
// (and, in its multi-token form, per short chunk of up to 8 new tokens per
// sequence, such as the verify step of speculative decoding).
//
// For every (sequence b, kv head, head group, split) CTA:
//   1. take pos, the slot of the (first) new token: from the launch parameters
//      (the cache's exact host copy of the lengths), or, in the variant built
//      for CUDA-graph capture, from the device lengths,
//   2. RMSNorm + RoPE the CTA's query rows (HPC <= 4 heads of the group, times
//      the new tokens in the multi-token form; at most 8 rows) at their
//      positions, rounded to bf16 like the prefill path, staged in shared memory,
//   3. the CTA owning the last split also norms + rotates the new tokens' k,
//      appends k' and v to their cache slots and attends to those new keys in
//      registers (token t sees new tokens 0..t),
//   4. stream its share of cache keys [0, pos) (or the attention window's part
//      of them) in 32-key chunks through a ring of shared-memory stages filled
//      by TMA tensor copies (128-byte swizzle, evict-first L2 policy), one
//      stage per consumer warp; all query rows of the CTA share every load,
//   5. per chunk and warp: S = q' K^T and O += P V as warp-level bf16 MMAs
//      (m16n8k16, fp32 accumulate; the query rows fill rows 0-7 of the 16-row
//      tile, so the tile's unused rows cost tensor time, not memory), online
//      softmax in fp32 on the score fragments, P reused in registers as the A
//      operand of P V,
//   6. the S split CTAs of a group form one thread-block cluster: each CTA
//      combines its consumer warps' partials in shared memory and pushes the
//      result (m, l, o) with st.async straight into the shared memory of the
//      CTA that owns each run of outputs, counted on that CTA's receive
//      mbarrier; each owner merges the S partials of its run in a fixed order
//      (deterministic) and writes the outputs in bf16; the length of b grows by
//      the new tokens (written by one CTA, or, with device lengths, by the last
//      group of the sequence through a counter).
// With programmatic dependent launch consecutive launches run side by side:
// a launch signals the next at its start and waits for the previous kernel
// only before loading the cache rows that a launch possibly still running
// appends to its layer (the host passes their number) and before its global
// writes.  The host plans the split count so that two launches' clusters fit
// on the device at once.
// This serves the decode step of the dryft-flash-infer agent guide ("Where the
// wins are": per-step overhead is the largest cost at batch 1 and 4, so the
// step is one launch) against the preallocated cache of the same section.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "qa.h"
#include "qa_device.cuh"

namespace qa {

constexpr int kK3Stages = kK3ConsumerWarps;  // one ring stage per consumer warp

// Floats a CTA receives in the split merge, maximised over the split count S:
// from each of the S CTAs of the cluster, an o run of E elements (E a multiple
// of 8) and (m, l) of every head.
constexpr int k3_recv_floats(int total, int hpc) {
    int best = 0;
    for (int S = 1; S <= kK3MaxSplits; ++S) {
        const int E = ((total + S - 1) / S + 7) & ~7;
        const int f = S * (E + 2 * hpc);
        best = f > best ? f : best;
    }
    return best;
}

// R = query rows of a CTA: HPC heads x TPS tokens (TPS = 1 for a decode step).
template <int D, int R>
struct K3Shape {
    static constexpr int kBoxBytes = kK3Chunk * 128;         // 32 rows x 64 bf16, swizzled
    static constexpr int kTileBytes = (D / 64) * kBoxBytes;  // K (or V) of one chunk
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kK3Stages * kStageBytes;
    static constexpr int kQBytes = (R * D * 2 + 15) & ~15;
    static constexpr int kRecvFloats = k3_recv_floats(R * D, R);
    static constexpr int kSmemBytes = 1024 + kRingBytes + kQBytes + kRecvFloats * 4;
    // Each consumer warp leaves its partial (o [row][D], then (m, l) [row][2])
    // in its own ring stage once it has consumed its last chunk.
    static_assert(R * (D + 2) * 4 <= kStageBytes, "partial must fit a ring stage");
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One gpu-scope acquire-release increment (publishes this thread's earlier
// writes and sees every earlier incrementer's).
__device__ __forceinline__ uint32_t atomic_inc_acq_rel(uint32_t *p) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
    return old;
}

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// RMSNorm + RoPE of one head row at one position, distributed over the D/8
// lanes of a row group (16 bytes each); cs holds (cos_a, sin_a, cos_b, sin_b)
// for this lane's 8 dims.  Returns the lane's 8 values as packed bf16.  Cast
// placement as in K1.
template <int D>
__device__ __forceinline__ uint4 norm_rope_row(const __nv_bfloat16 *src, const __nv_bfloat16 *w,
                                               const float4 (&cs)[4], float eps, int sub) {
    constexpr int LPR = D / 8, HALF = LPR / 2;
    const unsigned FULL = 0xffffffffu;
    const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(src) + sub);
    const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(w) + sub);
    float x[8], wf[8];
    unpack8(xv, x);
    unpack8(wv, wf);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
    for (int o = HALF; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
    const float r = rsqrtf(ss * (1.0f / D) + eps);
    uint32_t yw[4], pw[4], ow[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        yw[e] = pack_bf16(wf[2 * e] * round_bf16(x[2 * e] * r),
                          wf[2 * e + 1] * round_bf16(x[2 * e + 1] * r));
#pragma unroll
    for (int e = 0; e < 4; ++e) pw[e] = __shfl_xor_sync(FULL, yw[e], HALF);
    const bool lower = (sub % LPR) < HALF;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float y0 = bf16lo(yw[e]), y1 = bf16hi(yw[e]);
        const float q0 = bf16lo(pw[e]), q1 = bf16hi(pw[e]);
        const float r0 = lower ? y0 * cs[e].x - q0 * cs[e].y : y0 * cs[e].x + q0 * cs[e].y;
        const float r1 = lower ? y1 * cs[e].z - q1 * cs[e].w : y1 * cs[e].z + q1 * cs[e].w;
        ow[e] = pack_bf16(r0, r1);
    }
    return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// Byte offset of the 16-byte block db (8 bf16) of row `row` in a chunk tile:
// 64-column boxes of 32 rows x 128 bytes, 16-byte blocks XOR-swizzled by row.
__device__ __forceinline__ uint32_t swz(int row, int db) {
    return static_cast<uint32_t>((db >> 3) * (kK3Chunk * 128) + row * 128 +
                                 (((db & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t keep_pair(uint32_t x, bool lo, bool hi) {
    return (lo ? (x & 0x0000ffffu) : 0u) | (hi ? (x & 0xffff0000u) : 0u);
}

// One warp consumes one chunk of nk (1..32) keys whose K and V tiles start at
// shared addresses sK, sV.  Lane L owns query row L/4 of the MMA tile (rows
// 8..15 are padding); its score fragment covers keys nt*8 + 2(L%4) + {0,1}.
// The lane's row sees keys [klo, nk) of the chunk; kvlo <= klo of every row is
// the first key any row sees (rows below it, and from nk on, may hold anything).
template <int D>
__device__ __forceinline__ void consume_chunk(uint32_t sK, uint32_t sV, int nk, int klo, int kvlo,
                                              const uint32_t (&qa0)[D / 16],
                                              const uint32_t (&qa2)[D / 16], float c, float &m,
                                              float &l, float2 (&o)[D / 8], int lane) {
    const unsigned FULL = 0xffffffffu;
    const int mat = lane >> 3, r = lane & 7, q4 = lane & 3;
    float2 s[4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) s[nt] = make_float2(0.f, 0.f);
    // S = q' K^T: B fragments straight from the K rows (row = key, 8 dims per matrix row).
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int ntp = 0; ntp < 2; ++ntp) {
            const int key = (2 * ntp + (mat >> 1)) * 8 + r;
            uint32_t b[4];
            ldmatrix_x4(b, sK + swz(key, 2 * kk + (mat & 1)));
            mma_bf16_16816(s[2 * ntp], qa0[kk], qa2[kk], b[0], b[1]);
            mma_bf16_16816(s[2 * ntp + 1], qa0[kk], qa2[kk], b[2], b[3]);
        }
    }
    // Online softmax on the fragment (keys past nk, and before klo, are masked out).
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int k0 = nt * 8 + 2 * q4;
        if (k0 >= nk || k0 < klo) s[nt].x = -INFINITY;
        if (k0 + 1 >= nk || k0 + 1 < klo) s[nt].y = -INFINITY;
        mx = fmaxf(mx, fmaxf(s[nt].x, s[nt].y));
    }
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float alpha = (m == -INFINITY) ? 0.f : ex2((m - m_new) * c);
    const float neg = (m_new == -INFINITY) ? 0.f : m_new * c;  // a row with no key yet: p = 0
    float ps = 0.f;
    uint32_t pa[2][2];  // P as A fragments: [k-step][a0 | a2]
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const float p0 = ex2(fmaf(s[nt].x, c, -neg));
        const float p1 = ex2(fmaf(s[nt].y, c, -neg));
        ps += p0 + p1;
        pa[nt >> 1][nt & 1] = pack_bf16(p0, p1);
    }
    l = fmaf(l, alpha, ps);
    m = m_new;
    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt] = __fmul2_rn(o[nt], a2);
    // O += P V: B fragments from the V rows by transposing loads.  In a partial
    // chunk the rows outside [kvlo, nk) may hold anything (stale or poisoned, or
    // outside an attention window): drop them.
    const bool partial = nk < kK3Chunk || kvlo > 0;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
        for (int ndp = 0; ndp < D / 16; ++ndp) {
            const int key = ks * 16 + (mat & 1) * 8 + r;
            uint32_t b[4];
            ldmatrix_x4_trans(b, sV + swz(key, 2 * ndp + (mat >> 1)));
            if (partial) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int k0 = ks * 16 + (i & 1) * 8 + 2 * q4;
                    b[i] = keep_pair(b[i], k0 < nk && k0 >= kvlo, k0 + 1 < nk && k0 + 1 >= kvlo);
                }
            }
            mma_bf16_16816(o[2 * ndp], pa[ks][0], pa[ks][1], b[0], b[1]);
            mma_bf16_16816(o[2 * ndp + 1], pa[ks][0], pa[ks][1], b[2], b[3]);
        }
    }
}

// The kernel body.  A CTA serves the R = HPC x TPS query rows (token t, head
// h) -> row t * HPC + h of one (sequence, kv head, head group) for one split.
// TPS = 1 is the decode step: sequence b = b0 + blockIdx.z, one new token at
// slot pos[blockIdx.z] (launch parameters), or at lens[b] when kDevPos.
// TPS > 1 takes up to TPS new tokens of sequence mt->seq[blockIdx.z] at slots
// pos .. pos + ntok - 1: token t attends to the cache keys and to the new
// tokens 0..t (causal), and the cache takes all of them.
// kTableRope = true is the cache object's path: (cos, sin) from the library's
// table and the device length of b set after the step.  kTableRope = false is
// the allocation-free variant (TPS = 1): (cos, sin) of each sequence's
// position in cs_arr (cs_arr[blockIdx.z * D/2 + i]) and the caller keeps the
// lengths.  tmk / tmv: tensor maps (D, capacity, max_batch * Hkv) over this
// layer's K / V.
//
// Launches overlap the kernels before them on the stream (programmatic
// dependent launch).  With host positions a launch signals its dependents at
// once, and every CTA waits (griddepcontrol.wait) for the previous kernel
// before it exits; launches of this family still running when a launch starts
// may be writing cache rows of its layer just below its first new slot, and
// the host, which tracks them, passes their number as p.guard.  So before its
// own wait the body reads only its inputs (q, k, v, weights, rotary table)
// and the cache rows below pos - guard; the producer waits before loading the
// chunk holding that row, and every global write (cache slots, lengths, out)
// comes after a wait.  With device positions everything follows the wait and
// the signal comes right after it; the allocation-free variant (launched
// without overlap) never signals early.
template <int D, int HPC, int TPS, bool kTableRope, bool kDevPos>
__device__ __forceinline__ void k3_body(const K3Params &p, const float2 *cs_arr,
                                        const CUtensorMap *tmk, const CUtensorMap *tmv,
                                        const K3Multi *mt) {
    constexpr int R = HPC * TPS;
    static_assert(R <= 8, "query rows live in rows 0-7 of the MMA tile");
    static_assert(TPS == 1 || (kTableRope && !kDevPos), "multi-token steps use host positions");
    using Sh = K3Shape<D, R>;
    constexpr int LPR = D / 8;
    constexpr int NW = kK3ConsumerWarps;
    constexpr int NS = kK3Stages;
    const unsigned FULL = 0xffffffffu;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[NS], bar_empty[NS], bar_recv;
    __shared__ int s_abort;
    __shared__ __align__(16) __nv_bfloat16 s_newk[TPS * D], s_newv[TPS * D];  // new k', v
    __shared__ float s_w[R * kK3MaxSplits], s_linv[R];                         // merge weights

    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sRing = smem_u32(smem);
    __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(smem + Sh::kRingBytes);
    float *recv = reinterpret_cast<float *>(smem + Sh::kRingBytes + Sh::kQBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.HG, hg = blockIdx.y % p.HG;
    const int bl = blockIdx.z;
    const int b = TPS == 1 ? p.b0 + bl : mt->seq[bl];
    const int ntok = TPS == 1 ? 1 : mt->ntok[bl];
    const int qrow0 = TPS == 1 ? b : mt->row0[bl];  // row of token 0 in q, k, v, out
    // Host positions travel in the parameters; device positions are the lengths
    // an earlier kernel left: read here at once when they are settled (dev_pos
    // 2: the load's latency overlaps the set-up below), else after the launch
    // wait.  Every CTA of the sequence reads them before any writes them back.
    int pos = kDevPos ? (p.dev_pos == 2 ? p.lens[b] : 0) : p.pos[bl];
    const int S = p.S;

    // Merge geometry.  The CTA's R x D outputs are dealt to the S CTAs of the
    // cluster in runs of E (a multiple of 8); each of the NSRC = S CTAs (its
    // warps' partials combined first) sends the owner of each run its partial
    // o for the run and (m, l) of the rows the run touches.
    const int total = R * D;
    const int NSRC = S;
    const int E = ((total + S - 1) / S + 7) & ~7;
    const int e_lo = split * E;
    const int E_me = max(0, min(E, total - e_lo));
    const int g_lo = e_lo / D;
    const int nh_me = E_me > 0 ? (e_lo + E_me - 1) / D - g_lo + 1 : 0;
    float *rcv_o = recv;               // [NSRC][E]
    float *rcv_ml = recv + NSRC * E;   // [NSRC][R][2]

    // The cache chunks plus the new tokens (one unit, the last) are dealt to the
    // splits in shares that differ by one at most: split `split` streams chunks
    // [c_begin, c_end) and the last split also attends to the new tokens.
    bool pos_ok = false;
    int c_begin = 0, my_chunks = 0, c_safe = 0, first_round = 0, key_lo = 0, withheld = -1;
    auto plan = [&]() {
        pos_ok = pos >= 0 && ntok >= 1 && ntok <= TPS && pos + ntok <= p.cap;
        const int nchunks = pos_ok ? (pos + kK3Chunk - 1) / kK3Chunk : 0;
        // An attention window of W keys starts token t at key pos + t + 1 - W:
        // only the chunks from the one holding token 0's first key are streamed.
        key_lo = (pos_ok && p.window > 0) ? max(0, pos + 1 - p.window) : 0;
        const int c_lo = key_lo / kK3Chunk;
        const int64_t units = nchunks - c_lo + 1;
        c_begin = c_lo + static_cast<int>(split * units / S);
        const int c_end = c_lo + static_cast<int>(min((split + 1) * units / S,
                                                      static_cast<int64_t>(nchunks - c_lo)));
        my_chunks = max(0, c_end - c_begin);
        // chunks wholly below row pos - guard (all of them without a guard)
        c_safe = p.guard <= 0 ? nchunks : (pos > p.guard ? (pos - p.guard) / kK3Chunk : 0);
        first_round = min(NS, my_chunks);
        // Test hook (FaultPlan): every CTA of the first (sequence, kv head, head
        // group) cluster that streams cache chunks withholds its first one.
        withheld = (p.fault && blockIdx.y == 0 && blockIdx.z == 0 && my_chunks > 0) ? 0 : -1;
    };
    if (!kDevPos) plan();
    const bool owner = split == S - 1;
    const int64_t kv_base = static_cast<int64_t>(b) * p.seq_stride + kvh * p.head_stride;
    const int h_first = kvh * p.G + hg * HPC;  // first query head of this CTA
    const int tm_z = b * p.Hkv + kvh;          // (sequence, kv head) index in the tensor maps

    uint64_t policy = 0;
    // Stage `st` receives chunk c: K then V, each D/64 boxes of 32 rows.
    auto issue = [&](int c, int st) {
        if (c - c_begin == withheld) return;  // nothing completes this stage's phase
        const uint32_t fb = smem_u32(&bar_full[st]);
        mbar_expect_tx(fb, Sh::kStageBytes);
        const uint32_t dk = sRing + st * Sh::kStageBytes;
#pragma unroll
        for (int x = 0; x < D / 64; ++x) {
            tma_load_3d_hint(dk + x * Sh::kBoxBytes, tmk, x * 64, c * kK3Chunk, tm_z, fb, policy);
            tma_load_3d_hint(dk + Sh::kTileBytes + x * Sh::kBoxBytes, tmv, x * 64, c * kK3Chunk,
                             tm_z, fb, policy);
        }
    };
    int issued_early = 0;
    if (warp == NW && lane == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        mbar_init(smem_u32(&bar_recv), 1);
        prefetch_tmap(tmk);
        prefetch_tmap(tmv);
        s_abort = 0;
        if (E_me > 0) mbar_expect_tx(smem_u32(&bar_recv), NSRC * (E_me * 4 + nh_me * 8));
        fence_mbar_init();
        policy = policy_evict_first();
        // First loads at once, for the chunks no running kernel can be writing
        // (with host positions: device positions are not known yet).
        while (!kDevPos && issued_early < first_round && c_begin + issued_early < c_safe) {
            issue(c_begin + issued_early, issued_early);
            ++issued_early;
        }
    }
    cluster_arrive();  // peers may push into this CTA once they have waited on this

    // ---------------------------------------------------------------- prologue
    // The R query rows q' and, on the last split, the new tokens' k' and v go
    // to shared memory; all six warps share the rows (warp w takes items w,
    // w + 6, ...: query rows first, then new tokens) while the first loads are
    // in flight.  With host positions it runs before the launch wait, with
    // device positions after it.
    auto prologue = [&]() {
    if (pos_ok) {
        const int sub = lane % LPR;
        const int nitems = R + (owner ? ntok : 0);
        for (int it = warp; it < nitems; it += NW + 1) {  // warp-uniform
            const int t = it < R ? it / HPC : it - R;  // the item's token
            if (t >= ntok) continue;
            float4 cs[4];  // (cos_a, sin_a, cos_b, sin_b) of this lane's 8 dims at pos + t
            if constexpr (!kTableRope) {
                const float4 *src = reinterpret_cast<const float4 *>(cs_arr + bl * (D / 2) +
                                                                     8 * (sub % (LPR / 2)));
#pragma unroll
                for (int e = 0; e < 4; ++e) cs[e] = src[e];
            } else {
                const float4 *tab = reinterpret_cast<const float4 *>(
                    p.rope + static_cast<int64_t>(pos + t) * (D / 2) + 8 * (sub % (LPR / 2)));
#pragma unroll
                for (int e = 0; e < 4; ++e) cs[e] = __ldg(tab + e);
            }
            if (it < R) {
                const uint4 qp = norm_rope_row<D>(
                    p.q + (static_cast<int64_t>(qrow0 + t) * p.Hq + h_first + it % HPC) * D, p.wq,
                    cs, p.eps, sub);
                if (lane < LPR) reinterpret_cast<uint4 *>(qs + it * D)[sub] = qp;
            } else {
                // A new token: k' and v; the copy into cache slot pos + t waits for
                // the previous kernel below.
                const int64_t kr = (static_cast<int64_t>(qrow0 + t) * p.Hkv + kvh) * D;
                const uint4 kp = norm_rope_row<D>(p.k + kr, p.wk, cs, p.eps, sub);
                const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(p.v + kr) + sub);
                if (lane < LPR) {
                    reinterpret_cast<uint4 *>(s_newk + t * D)[sub] = kp;
                    reinterpret_cast<uint4 *>(s_newv + t * D)[sub] = vv;
                }
            }
        }
    }
    };
    // Programmatic dependent launch: griddepcontrol.wait (the previous kernel
    // has finished and its writes are visible) is executed only where this step
    // depends on it: with host positions, before loading the chunk holding row
    // pos - guard and before every global write; with device positions, before
    // reading them.  Every CTA passes a wait before it exits.
    if constexpr (!kDevPos) {
        if constexpr (kTableRope) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        prologue();
    } else {
        if (p.dev_pos == 2) {
            // No launch that may still run writes this layer (the host's launch
            // record says so): its lengths are settled (read above) and the step
            // proceeds as one with host positions, signalling the next launch at
            // once.
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            plan();
            if (warp == NW && lane == 0) {
                for (; issued_early < first_round && c_begin + issued_early < c_safe; ++issued_early)
                    issue(c_begin + issued_early, issued_early);
            }
        } else {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            pos = p.lens[b];
            plan();
            if (warp == NW && lane == 0) {
                for (; issued_early < first_round; ++issued_early)
                    issue(c_begin + issued_early, issued_early);
            }
        }
        prologue();
    }
    if (!pos_ok) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (threadIdx.x == 0) set_error(p.err, kErrBounds, kKernK3, 1);
        return;
    }
    __syncthreads();  // ring initialised, q' and the new tokens in shared memory

    if (warp == NW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool waited = kDevPos && p.dev_pos != 2;
            int issued = issued_early;
            for (; issued < my_chunks; ++issued) {
                const int st = issued % NS;
                if (issued >= NS &&
                    !mbar_wait(smem_u32(&bar_empty[st]), ((issued / NS) - 1) & 1, &s_abort, p.err,
                               kKernK3, 2, p.wait_ns))
                    break;
                if (!waited && c_begin + issued >= c_safe) {  // may hold a previous step's rows
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    waited = true;
                }
                issue(c_begin + issued, st);
            }
            // No copy may land after the CTA exits: wait (bounded) for the last ones.
            for (int i = max(0, issued - NS); i < issued; ++i) {
                if (i == withheld) continue;
                int dummy = 0;
                mbar_wait(smem_u32(&bar_full[i % NS]), (i / NS) & 1, &dummy, p.err, kKernK3, 3, p.wait_ns);
            }
        }

    } else {
        // ------------------------------------------------------------ consumers
        // A fragments of q' (row r = lane / 4 of the 16-row tile; padding rows zero).
        const int hrow = lane >> 2, q4 = lane & 3;
        const int trow = TPS == 1 ? 0 : hrow / HPC;  // the row's token
        const bool real = hrow < R && trow < ntok;
        uint32_t qa0[D / 16], qa2[D / 16];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(qs + hrow * D + 16 * kk);
            qa0[kk] = real ? qrow[q4] : 0u;
            qa2[kk] = real ? qrow[4 + q4] : 0u;
        }
        // First cache key of the row's window: token t at pos + t sees keys from
        // pos + t + 1 - W.
        const int row_lo = p.window > 0 ? max(0, pos + trow + 1 - p.window) : 0;
        float m = -INFINITY, l = 0.f;
        float2 o[D / 8];
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) o[nt] = make_float2(0.f, 0.f);

        for (int c = c_begin + warp, i = warp; i < my_chunks; c += NW, i += NW) {
            const int st = i % NS;
            bool ok = mbar_wait(smem_u32(&bar_full[st]), (i / NS) & 1, &s_abort, p.err, kKernK3, 4, p.wait_ns);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            const int base = c * kK3Chunk;
            const int nk = min(kK3Chunk, pos - base);
            const uint32_t sk = sRing + st * Sh::kStageBytes;
            const int kvlo = max(0, key_lo - base);
            const int klo = TPS == 1 ? kvlo : min(kK3Chunk, max(0, row_lo - base));
            consume_chunk<D>(sk, sk + Sh::kTileBytes, nk, klo, kvlo, qa0, qa2, p.scale_log2, m, l,
                             o, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_empty[st]));
        }
        if (owner && warp == my_chunks % NW) {
            // The new tokens, on the warp whose turn is next: s_u = q'.k'_u (the 4
            // lanes of a row split the dims) for the tokens u <= t the row's token
            // t sees (and, with a window of W keys, t - u < W), then one
            // online-softmax update of the lane's o.
            const float c = p.scale_log2;
            float sd[TPS];
            float mx = -INFINITY;
#pragma unroll
            for (int u = 0; u < TPS; ++u) {
                float x = 0.f;
                if (real && u <= trow) {
                    const __nv_bfloat162 *qh =
                        reinterpret_cast<const __nv_bfloat162 *>(qs + hrow * D) + q4 * (D / 8);
                    const __nv_bfloat162 *kh =
                        reinterpret_cast<const __nv_bfloat162 *>(s_newk + u * D) + q4 * (D / 8);
#pragma unroll
                    for (int i = 0; i < D / 8; ++i) {
                        const float2 a = __bfloat1622float2(qh[i]), kk = __bfloat1622float2(kh[i]);
                        x = fmaf(a.x, kk.x, fmaf(a.y, kk.y, x));
                    }
                }
                x += __shfl_xor_sync(FULL, x, 1);
                x += __shfl_xor_sync(FULL, x, 2);
                const bool seen = real && u <= trow && (p.window <= 0 || trow - u < p.window);
                sd[u] = seen ? x : -INFINITY;
                mx = fmaxf(mx, sd[u]);
            }
            const float m_new = fmaxf(m, mx);
            const float alpha = (m == -INFINITY) ? 0.f : ex2((m - m_new) * c);
            const float neg = (m_new == -INFINITY) ? 0.f : m_new * c;
            float pn[TPS], ps = 0.f;
#pragma unroll
            for (int u = 0; u < TPS; ++u) {
                pn[u] = ex2(fmaf(sd[u], c, -neg));
                ps += pn[u];
            }
            l = fmaf(l, alpha, q4 == 0 ? ps : 0.f);  // l is summed over the quad below
            m = m_new;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                float2 acc = make_float2(o[nt].x * alpha, o[nt].y * alpha);
#pragma unroll
                for (int u = 0; u < TPS; ++u) {
                    if (u < ntok) {
                        const float2 vv = __bfloat1622float2(
                            reinterpret_cast<const __nv_bfloat162 *>(s_newv + u * D)[nt * 4 + q4]);
                        acc = make_float2(fmaf(pn[u], vv.x, acc.x), fmaf(pn[u], vv.y, acc.y));
                    }
                }
                o[nt] = acc;
            }
        }
        l += __shfl_xor_sync(FULL, l, 1);
        l += __shfl_xor_sync(FULL, l, 2);

        // The warp's partial into its own ring stage (no copy lands there any
        // more): lane (hrow, q4) holds o[hrow][nt*8 + 2*q4 + {0,1}] and (m, l)
        // of row hrow.
        if (real) {
            float *red = reinterpret_cast<float *>(smem + warp * Sh::kStageBytes);
            float *dst = red + hrow * D;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt)
                *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * q4) = o[nt];
            if (q4 == 0) {
                red[R * D + hrow * 2] = m;
                red[R * D + hrow * 2 + 1] = l;
            }
        }
    }

    // ---------------------------------------------------------------- combine and push
    // The NW warp partials of the CTA become one (m, l, o) per row, in a fixed
    // order; each pair of outputs goes to the CTA owning its run, (m, l) of a
    // row to every owner whose run touches the row.  Rows of tokens past ntok
    // are carried along and never written out.
    __syncthreads();
    cluster_wait();  // every peer's receive barrier is initialised
    {
        const float c = p.scale_log2;
        constexpr int kWF = Sh::kStageBytes / 4;  // floats between two warps' partials
        const float *red = reinterpret_cast<const float *>(smem);
        const uint32_t a_bar = smem_u32(&bar_recv);
        const uint32_t a_o = smem_u32(rcv_o + split * E);
        for (int pe = threadIdx.x; pe < total / 2; pe += blockDim.x) {
            const int e = 2 * pe, g = e / D, d = e % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, red[w * kWF + R * D + g * 2]);
            float2 O = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float mw = red[w * kWF + R * D + g * 2];
                const float wt = mw == -INFINITY ? 0.f : ex2((mw - M) * c);
                const float2 ow = *reinterpret_cast<const float2 *>(red + w * kWF + g * D + d);
                O = make_float2(fmaf(wt, ow.x, O.x), fmaf(wt, ow.y, O.y));
            }
            const int dst = e / E;
            st_async_f32x2(map_rank(a_o + 4u * (e - dst * E), dst), O.x, O.y, map_rank(a_bar, dst));
        }
        for (int k = threadIdx.x; k < R * S; k += blockDim.x) {
            const int g = k / S, dst = k % S;
            const int lo = dst * E, hi = min(lo + E, total);
            if (lo < hi && lo < (g + 1) * D && hi > g * D) {
                float M = -INFINITY, Lsum = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) M = fmaxf(M, red[w * kWF + R * D + g * 2]);
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float mw = red[w * kWF + R * D + g * 2];
                    if (mw != -INFINITY)
                        Lsum = fmaf(ex2((mw - M) * c), red[w * kWF + R * D + g * 2 + 1], Lsum);
                }
                st_async_f32x2(map_rank(smem_u32(rcv_ml + (split * R + g) * 2), dst), M, Lsum,
                               map_rank(a_bar, dst));
            }
        }
    }

    // ---------------------------------------------------------------- merge
    // Once every source's bytes have landed: per row of the run (one warp
    // each), w_i = 2^((m_i - M) c) with M = max_i m_i and 1 / sum_i w_i l_i;
    // then each output of the run is sum_i w_i o_i times that, over the sources
    // in a fixed order (deterministic).  The merge reads only this cluster's
    // shared memory, so it runs before the launch wait, and only the global
    // writes (cache slots, lengths, outputs) follow the wait: the part of a step
    // that waits for the previous kernel's end is a few stores.
    constexpr int kThreadsK3 = (NW + 1) * 32;
    constexpr int kOutPer = (R * D + kThreadsK3 - 1) / kThreadsK3;  // outputs per thread, at most
    float res[kOutPer];
    bool merged = E_me > 0;
    if (E_me > 0) {
        bool ok = mbar_wait_cluster(smem_u32(&bar_recv), 0, &s_abort, p.err, kKernK3, 5, p.wait_ns);
        if (!ok) {
            // Given up (this CTA timed out somewhere): the peers still push their
            // partials here, so every inbound st.async must land before this CTA
            // exits and its shared memory goes away.  Bounded like every wait.
            int dummy = 0;
            mbar_wait_cluster(smem_u32(&bar_recv), 0, &dummy, p.err, kKernK3, 6, p.wait_ns);
        }
        merged = __syncthreads_and(ok);
        if (merged) {
            const float c = p.scale_log2;
            constexpr int kPerLane = (kK3MaxSplits + 31) / 32;
            for (int hl = warp; hl < nh_me; hl += NW + 1) {
                const float *ml = rcv_ml + 2 * (g_lo + hl);  // source i: ml[2 * R * i], l after it
                float mi[kPerLane], M = -INFINITY;
#pragma unroll
                for (int k = 0; k < kPerLane; ++k) {
                    const int i = lane + 32 * k;
                    mi[k] = i < NSRC ? ml[2 * R * i] : -INFINITY;
                    M = fmaxf(M, mi[k]);
                }
#pragma unroll
                for (int o2 = 16; o2 >= 1; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o2));
                float Ls = 0.f;
#pragma unroll
                for (int k = 0; k < kPerLane; ++k) {
                    const int i = lane + 32 * k;
                    if (i < NSRC) {
                        const float w = mi[k] == -INFINITY ? 0.f : ex2((mi[k] - M) * c);
                        s_w[hl * kK3MaxSplits + i] = w;
                        Ls = fmaf(w, ml[2 * R * i + 1], Ls);
                    }
                }
#pragma unroll
                for (int o2 = 16; o2 >= 1; o2 >>= 1) Ls += __shfl_xor_sync(FULL, Ls, o2);
                if (lane == 0) s_linv[hl] = 1.f / Ls;
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < kOutPer; ++j) {
                const int k = threadIdx.x + j * kThreadsK3;
                res[j] = 0.f;
                if (k < E_me) {
                    const int e = e_lo + k, g = e / D, hl = g - g_lo;
                    const float *w = s_w + hl * kK3MaxSplits;
                    const float *src = rcv_o + k;
                    float O4[4] = {0.f, 0.f, 0.f, 0.f};  // four running sums, in a fixed order
                    int i = 0;
                    for (; i + 4 <= NSRC; i += 4) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) O4[u] = fmaf(w[i + u], src[(i + u) * E], O4[u]);
                    }
                    for (; i < NSRC; ++i) O4[0] = fmaf(w[i], src[i * E], O4[0]);
                    res[j] = ((O4[0] + O4[1]) + (O4[2] + O4[3])) * s_linv[hl];
                }
            }
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // before any global write below
    if (owner && hg == 0 && warp == NW && lane < LPR) {
        // Slots pos.. of the cache, read only by later launches.
        for (int t = 0; t < ntok; ++t) {
            reinterpret_cast<uint4 *>(p.kc + kv_base + static_cast<int64_t>(pos + t) * D)[lane] =
                reinterpret_cast<const uint4 *>(s_newk + t * D)[lane];
            reinterpret_cast<uint4 *>(p.vc + kv_base + static_cast<int64_t>(pos + t) * D)[lane] =
                reinterpret_cast<const uint4 *>(s_newv + t * D)[lane];
        }
    }
    if constexpr (kTableRope && !kDevPos) {
        if (split == 0 && blockIdx.y == 0 && threadIdx.x == 0) p.lens[b] = pos + ntok;
    }
    if (!merged) return;
    if (kDevPos && split == 0 && threadIdx.x == 0) {
        // Every CTA of this group has pushed, so it has read lens[b]: count the
        // group towards sequence b; the last group of the sequence advances it.
        const uint32_t prev = atomic_inc_acq_rel(p.seq_cnt + b);
        if (prev == static_cast<uint32_t>(p.Hkv * p.HG) - 1u) {
            p.lens[b] = pos + 1;
            p.seq_cnt[b] = 0u;
        }
    }
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) {
        const int k = threadIdx.x + j * kThreadsK3;
        if (k < E_me) {
            const int e = e_lo + k, g = e / D, d = e % D;
            const int t = g / HPC, hh = g % HPC;
            if (t < ntok)
                p.out[(static_cast<int64_t>(qrow0 + t) * p.Hq + h_first + hh) * D + d] =
                    __float2bfloat16_rn(res[j]);
        }
    }
}

template <int D, int HPC, bool kDevPos>
__global__ void __launch_bounds__((kK3ConsumerWarps + 1) * 32, 2)
    k3_decode_kernel(const __grid_constant__ K3Params p) {
    k3_body<D, HPC, 1, true, kDevPos>(p, nullptr, &p.tmk, &p.tmv, nullptr);
}

// Up to TPS new tokens per sequence (HPC x TPS = 8 query rows per CTA).
struct K3MultiParams {
    K3Params base;
    K3Multi mt;
};

template <int D, int HPC, int TPS>
__global__ void __launch_bounds__((kK3ConsumerWarps + 1) * 32, 2)
    k3_multi_kernel(const __grid_constant__ K3MultiParams p) {
    k3_body<D, HPC, TPS, true, false>(p.base, nullptr, &p.base.tmk, &p.base.tmv, &p.mt);
}

template <int D, int HPC, bool kDevPos>
static cudaError_t launch_k3_t(const K3Params &p, cudaStream_t stream) {
    constexpr int smem = K3Shape<D, HPC>::kSmemBytes;
    static std::atomic<unsigned> configured{0u};  // devices 0..31 set up (one bit each)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 32 || !((configured.load(std::memory_order_acquire) >> dev) & 1u)) {
        cudaError_t e = cudaFuncSetAttribute(k3_decode_kernel<D, HPC, kDevPos>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k3_decode_kernel<D, HPC, kDevPos>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        if (dev < 32) configured.fetch_or(1u << dev, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.S, p.Hkv * p.HG, p.B);
    cfg.blockDim = dim3((kK3ConsumerWarps + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;  // one cluster = the splits of a group
    attr[0].val.clusterDim.x = p.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k3_decode_kernel<D, HPC, kDevPos>, p);
}

template <typename Kern>
static int cluster_capacity_k(Kern kern, int smem, int S) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3((kK3ConsumerWarps + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int D, int HPC>
static int cluster_capacity_t(int S, bool multi) {
    if (!multi) return cluster_capacity_k(k3_decode_kernel<D, HPC, false>, K3Shape<D, HPC>::kSmemBytes, S);
    return cluster_capacity_k(k3_multi_kernel<D, HPC, 8 / HPC>, K3Shape<D, 8>::kSmemBytes, S);
}

// Per device, head_dim, form and heads per CTA: the capacity for every S,
// queried once ([S], 0 = query failed).  The table is filled under the lock and
// never changes afterwards, so callers read it without locking.
static const int *capacity_table(int D, int HPC, bool multi) {
    constexpr int kDev = 16;
    struct Table {
        std::atomic<bool> ready{false};
        int cap[kK3MaxSplits + 1] = {};
    };
    static Table tables[kDev][2][2][3];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDev) return nullptr;
    if ((D != 64 && D != 128) || (HPC != 1 && HPC != 2 && HPC != 4)) return nullptr;
    Table &t = tables[dev][D == 128 ? 1 : 0][multi ? 1 : 0][HPC == 4 ? 2 : (HPC == 2 ? 1 : 0)];
    if (!t.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(mu);
        if (!t.ready.load(std::memory_order_relaxed)) {
            for (int S = 1; S <= kK3MaxSplits; ++S) {
                int n = 0;
                if (D == 128)
                    n = HPC == 4 ? cluster_capacity_t<128, 4>(S, multi)
                                 : (HPC == 2 ? cluster_capacity_t<128, 2>(S, multi)
                                             : cluster_capacity_t<128, 1>(S, multi));
                else
                    n = HPC == 4 ? cluster_capacity_t<64, 4>(S, multi)
                                 : (HPC == 2 ? cluster_capacity_t<64, 2>(S, multi)
                                             : cluster_capacity_t<64, 1>(S, multi));
                t.cap[S] = n > 0 ? n : 0;
            }
            t.ready.store(true, std::memory_order_release);
        }
    }
    return t.cap;
}

int k3_cluster_capacity(int D, int HPC, int S, bool multi) {
    if (S < 1 || S > kK3MaxSplits) return 0;
    const int *cap = capacity_table(D, HPC, multi);
    return cap ? cap[S] : 0;
}

template <typename Kern>
static int occupancy_k(Kern kern, int smem) {
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, (kK3ConsumerWarps + 1) * 32, smem) !=
            cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return n;
}

template <int D>
static int max_occupancy_d() {
    const int v[] = {
        occupancy_k(k3_decode_kernel<D, 1, false>, K3Shape<D, 1>::kSmemBytes),
        occupancy_k(k3_decode_kernel<D, 2, false>, K3Shape<D, 2>::kSmemBytes),
        occupancy_k(k3_decode_kernel<D, 4, false>, K3Shape<D, 4>::kSmemBytes),
        occupancy_k(k3_decode_kernel<D, 1, true>, K3Shape<D, 1>::kSmemBytes),
        occupancy_k(k3_decode_kernel<D, 2, true>, K3Shape<D, 2>::kSmemBytes),
        occupancy_k(k3_decode_kernel<D, 4, true>, K3Shape<D, 4>::kSmemBytes),
        occupancy_k(k3_multi_kernel<D, 1, 8>, K3Shape<D, 8>::kSmemBytes),
        occupancy_k(k3_multi_kernel<D, 2, 4>, K3Shape<D, 8>::kSmemBytes),
        occupancy_k(k3_multi_kernel<D, 4, 2>, K3Shape<D, 8>::kSmemBytes)};
    int best = 0;
    for (int x : v) {
        if (x < 0) return -1;
        best = std::max(best, x);
    }
    return best;
}

int k3_max_resident_ctas() {
    constexpr int kDev = 64;
    static std::atomic<int> cache[kDev] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return 1 << 20;
    }
    if (dev < kDev) {
        const int known = cache[dev].load(std::memory_order_acquire);
        if (known > 0) return known;
    }
    int sms = 0, per_sm_limit = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm_limit, cudaDevAttrMaxBlocksPerMultiprocessor, dev) !=
            cudaSuccess) {
        cudaGetLastError();
        return 1 << 20;
    }
    if (dev >= kDev) return sms * per_sm_limit;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].load(std::memory_order_relaxed) == 0) {
        const int a = max_occupancy_d<64>(), b = max_occupancy_d<128>();
        // a failed query falls back to the architectural limit of CTAs per SM
        const int per_sm = (a < 0 || b < 0) ? per_sm_limit : std::max(std::max(a, b), 1);
        cache[dev].store(sms * per_sm, std::memory_order_release);
    }
    return cache[dev].load(std::memory_order_relaxed);
}

int k3_choose_splits(int D, int HPC, int groups, int pos_max, bool multi, int overlap) {
    const int nchunks = (pos_max + kK3Chunk - 1) / kK3Chunk;
    const int64_t need = static_cast<int64_t>(std::max(overlap, 1)) * groups;
    const int *cap = capacity_table(D, HPC, multi);
    int best = 1;
    if (!cap) return best;
    for (int S = 2; S <= std::min(kK3MaxSplits, std::max(1, nchunks)); ++S)
        if (cap[S] >= need) best = S;
    return best;
}

template <bool kDevPos>
static cudaError_t launch_k3_d(const K3Params &p, int D, int HPC, cudaStream_t stream) {
    if (D == 128) {
        if (HPC == 4) return launch_k3_t<128, 4, kDevPos>(p, stream);
        if (HPC == 2) return launch_k3_t<128, 2, kDevPos>(p, stream);
        if (HPC == 1) return launch_k3_t<128, 1, kDevPos>(p, stream);
    } else if (D == 64) {
        if (HPC == 4) return launch_k3_t<64, 4, kDevPos>(p, stream);
        if (HPC == 2) return launch_k3_t<64, 2, kDevPos>(p, stream);
        if (HPC == 1) return launch_k3_t<64, 1, kDevPos>(p, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_k3(const K3Params &p, int D, int HPC, cudaStream_t stream) {
    return p.dev_pos ? launch_k3_d<true>(p, D, HPC, stream) : launch_k3_d<false>(p, D, HPC, stream);
}

template <int D, int HPC>
static cudaError_t launch_k3_multi_t(const K3MultiParams &p, cudaStream_t stream) {
    constexpr int TPS = 8 / HPC;
    constexpr int smem = K3Shape<D, 8>::kSmemBytes;
    auto kern = k3_multi_kernel<D, HPC, TPS>;
    static std::atomic<unsigned> configured{0u};  // devices 0..31 set up (one bit each)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 32 || !((configured.load(std::memory_order_acquire) >> dev) & 1u)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        if (dev < 32) configured.fetch_or(1u << dev, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.base.S, p.base.Hkv * p.base.HG, p.base.B);
    cfg.blockDim = dim3((kK3ConsumerWarps + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.base.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_k3_multi(const K3Params &p, const K3Multi &m, int D, int HPC,
                            cudaStream_t stream) {
    K3MultiParams mp;
    mp.base = p;
    mp.mt = m;
    if (D == 128) {
        if (HPC == 4) return launch_k3_multi_t<128, 4>(mp, stream);
        if (HPC == 2) return launch_k3_multi_t<128, 2>(mp, stream);
        if (HPC == 1) return launch_k3_multi_t<128, 1>(mp, stream);
    } else if (D == 64) {
        if (HPC == 4) return launch_k3_multi_t<64, 4>(mp, stream);
        if (HPC == 2) return launch_k3_multi_t<64, 2>(mp, stream);
        if (HPC == 1) return launch_k3_multi_t<64, 1>(mp, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qa

// ==================================================================== allocation-free decode step
// qa_decode_step_noalloc runs the same decode kernel body for callers that may
// not allocate device memory.  The kernel's global scratch lives in a fixed
// array of this module: the CUDA driver creates it when the library's device
// code loads on a GPU, and it stays until the process exits.  Host code never
// dereferences the symbol; it asks the runtime for the array's device address
// once per device.  (The splits are merged in distributed shared memory, so
// the array holds the error word only.)
namespace qa {

constexpr size_t kNoAllocScratchBytes = 256;
constexpr int kNoAllocMaxBatch = 16;
static_assert(kNoAllocMaxBatch <= kK3MaxSeqPerLaunch, "positions travel in K3Params::pos");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct alignas(64) K3NoAllocParams {
    K3Params base;                     // base.tmk / tmv over the caller's K / V of this layer;
                                       // base.pos[b]: slot of each sequence's new token
    float2 cs[kNoAllocMaxBatch * 64];  // (cos, sin) at pos[b] of the D/2 frequencies, [b][i]
};

template <int D, int HPC>
__global__ void __launch_bounds__((kK3ConsumerWarps + 1) * 32, 2)
    k3_decode_noalloc_kernel(const __grid_constant__ K3NoAllocParams p) {
    k3_body<D, HPC, 1, false, false>(p.base, p.cs, &p.base.tmk, &p.base.tmv, nullptr);
}

template <int D, int HPC>
static cudaError_t launch_noalloc_t(const K3NoAllocParams &p, cudaStream_t stream) {
    constexpr int smem = K3Shape<D, HPC>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(k3_decode_noalloc_kernel<D, HPC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k3_decode_noalloc_kernel<D, HPC>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.base.S, p.base.Hkv * p.base.HG, p.base.B);
    cfg.blockDim = dim3((kK3ConsumerWarps + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.base.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k3_decode_noalloc_kernel<D, HPC>, p);
}

static cudaError_t launch_noalloc(const K3NoAllocParams &p, int D, int HPC, cudaStream_t stream) {
    if (D == 128) {
        if (HPC == 4) return launch_noalloc_t<128, 4>(p, stream);
        if (HPC == 2) return launch_noalloc_t<128, 2>(p, stream);
        if (HPC == 1) return launch_noalloc_t<128, 1>(p, stream);
    } else if (D == 64) {
        if (HPC == 4) return launch_noalloc_t<64, 4>(p, stream);
        if (HPC == 2) return launch_noalloc_t<64, 2>(p, stream);
        if (HPC == 1) return launch_noalloc_t<64, 1>(p, stream);
    }
    return cudaErrorInvalidValue;
}

namespace {
struct NoAllocDevice {
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];

// Once per device, with that device current: the device address of the
// scratch array and the SM count.  Neither call allocates.
qa_status noalloc_setup(NoAllocDevice *&out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
        return QA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc_devices[dev];
    if (!d.scratch) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return QA_ERR_CUDA;
        }
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return QA_ERR_CUDA;
        d.num_sms = sms;
        d.scratch = static_cast<unsigned char *>(ptr);
    }
    out = &d;
    return QA_OK;
}

bool aligned16_na(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace
}  // namespace qa

extern "C" __attribute__((visibility("default"))) qa_status qa_decode_step_noalloc(
    const qa_config *cfg, int batch, const int32_t *positions, void *k_cache, void *v_cache,
    const void *q, const void *k, const void *v, const void *q_norm_w, const void *k_norm_w,
    void *out, void *stream) {
    using namespace qa;
    if (!cfg || !positions) return QA_ERR_INVALID_ARG;
    const qa_config g = *cfg;
    if (g.max_batch <= 0 || g.capacity <= 0 || !(g.rope_theta > 0.f) || !(g.rms_eps >= 0.f))
        return QA_ERR_INVALID_ARG;
    if ((g.head_dim != 64 && g.head_dim != 128) || g.n_kv_heads <= 0 || g.n_q_heads <= 0 ||
        g.n_q_heads % g.n_kv_heads)
        return QA_ERR_UNSUPPORTED_SHAPE;
    const int G = g.n_q_heads / g.n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return QA_ERR_UNSUPPORTED_SHAPE;
    if (batch < 1 || batch > g.max_batch) return QA_ERR_INVALID_ARG;
    if (batch > kNoAllocMaxBatch) return QA_ERR_UNSUPPORTED_SHAPE;  // above the parameter block
    if (!k_cache || !v_cache || !q || !k || !v || !q_norm_w || !k_norm_w || !out)
        return QA_ERR_INVALID_ARG;
    if (!aligned16_na(k_cache) || !aligned16_na(v_cache) || !aligned16_na(q) ||
        !aligned16_na(k) || !aligned16_na(v) || !aligned16_na(q_norm_w) ||
        !aligned16_na(k_norm_w) || !aligned16_na(out))
        return QA_ERR_ALIGNMENT;
    int pos_max = 0;
    for (int b = 0; b < batch; ++b) {
        if (positions[b] < 0) return QA_ERR_INVALID_ARG;
        if (positions[b] >= g.capacity) return QA_ERR_CAPACITY;  // no slot left: never evict
        pos_max = std::max(pos_max, static_cast<int>(positions[b]));
    }
    const int HPC = std::min(G, 4), HG = G / HPC, D = g.head_dim;
    const int groups = batch * g.n_kv_heads * HG;
    if (g.n_kv_heads * HG > 65535) return QA_ERR_UNSUPPORTED_SHAPE;
    NoAllocDevice *dev = nullptr;
    qa_status st = noalloc_setup(dev);
    if (st != QA_OK) return st;

    // Split plan as in qa_decode_step (the variant has the same resources).
    // (launched without overlap: the clusters of one step are enough)
    const int S = k3_choose_splits(D, HPC, groups, pos_max, false, 1);

    K3NoAllocParams p{};
    if (!encode_decode_map(&p.base.tmk, k_cache, D, g.capacity, g.max_batch * g.n_kv_heads) ||
        !encode_decode_map(&p.base.tmv, v_cache, D, g.capacity, g.max_batch * g.n_kv_heads))
        return QA_ERR_CUDA;
    for (int b = 0; b < batch; ++b) {
        p.base.pos[b] = positions[b];
        for (int i = 0; i < D / 2; ++i) {  // same fp64 formula as the cache's table
            const double a = static_cast<double>(positions[b]) *
                             std::pow(static_cast<double>(g.rope_theta), -2.0 * i / D);
            p.cs[b * (D / 2) + i] =
                make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
        }
    }
    unsigned char *scr = dev->scratch;
    K3Params &bp = p.base;
    bp.q = static_cast<const __nv_bfloat16 *>(q);
    bp.k = static_cast<const __nv_bfloat16 *>(k);
    bp.v = static_cast<const __nv_bfloat16 *>(v);
    bp.wq = static_cast<const __nv_bfloat16 *>(q_norm_w);
    bp.wk = static_cast<const __nv_bfloat16 *>(k_norm_w);
    bp.kc = static_cast<__nv_bfloat16 *>(k_cache);
    bp.vc = static_cast<__nv_bfloat16 *>(v_cache);
    bp.lens = nullptr;
    bp.rope = nullptr;
    bp.err = reinterpret_cast<uint32_t *>(scr);
    bp.out = static_cast<__nv_bfloat16 *>(out);
    bp.head_stride = static_cast<int64_t>(g.capacity) * D;
    bp.seq_stride = bp.head_stride * g.n_kv_heads;
    bp.b0 = 0;
    bp.dev_pos = 0;
    bp.seq_cnt = nullptr;
    bp.window = 0;
    bp.guard = 0;  // launched without overlap: the previous kernel has finished
    bp.B = batch;
    bp.Hq = g.n_q_heads;
    bp.Hkv = g.n_kv_heads;
    bp.G = G;
    bp.HG = HG;
    bp.cap = g.capacity;
    bp.S = S;
    bp.eps = g.rms_eps;
    bp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    const FaultPlan f = take_fault(QA_KERNEL_DECODE_ATTN);
    bp.fault = f.fault;
    bp.wait_ns = f.wait_ns;

    // The error word is zero when the library loads and after every read
    // through qa_noalloc_get_device_error; a call does not clear it, so the
    // first error of any call since the last read is kept for the caller.
    if (launch_noalloc(p, D, HPC, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return QA_ERR_CUDA;
    return QA_OK;
}

extern "C" __attribute__((visibility("default"))) qa_status qa_noalloc_get_device_error(
    uint32_t *detail, void *stream) {
    using namespace qa;
    NoAllocDevice *dev = nullptr;
    qa_status st = noalloc_setup(dev);
    if (st != QA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    // A copy into this stack word and a 4-byte memset: neither allocates.
    if (cudaMemcpyAsync(&word, dev->scratch, sizeof(word), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return QA_ERR_CUDA;
    if (word != 0 && (cudaMemsetAsync(dev->scratch, 0, sizeof(word), s) != cudaSuccess ||
                      cudaStreamSynchronize(s) != cudaSuccess))
        return QA_ERR_CUDA;
    if (detail) *detail = word;
    switch (word & 0xffu) {
        case 0: return QA_OK;
        case kErrTimeout: return QA_ERR_DEVICE_TIMEOUT;
        default: return QA_ERR_DEVICE_BOUNDS;
    }
}
