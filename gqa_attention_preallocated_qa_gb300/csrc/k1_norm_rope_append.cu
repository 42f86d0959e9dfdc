// k1_norm_rope_append.cu -- K1: fused per-head QK-RMSNorm + rotary embedding +
// KV-cache append for the rows of a prefill.
//
// "RMSNorm, rotary embedding ... are small, repeated, and safe to fuse"
// (dryft-flash-infer agent guide, "Where the wins are", fused-kernels bullet);
// "a preallocated, correctly strided cache removes per-step allocation and
// concatenation" (same section, KV-cache-layout bullet).
//
// One head row (D bf16 = D*2 bytes) is handled by D/8 lanes, 16 bytes each:
// 128-bit coalesced loads and stores, the sum of squares reduced with warp
// shuffles, the rotate-half partner (dimension d +- D/2) fetched with one more
// shuffle.  Rows of a token are q heads, then k heads, then v heads; a v row
// is copied bit-exactly.
//
// Cast placement of the RMSNorm follows the Qwen3 module the guide's numerics
// section points at: the normalised vector is rounded to bf16 before the
// weight multiply, and the product is rounded to bf16 again.  RoPE is then
// computed in fp32 from an fp64-derived (cos, sin) table and rounded once.
#include <algorithm>
#include <atomic>

#include "qa_device.cuh"

namespace qa {

cudaError_t launch_k1_rows(const K1Params &p, int D, cudaStream_t stream);

// Head rows handled by one row group (LPR lanes): all their loads are issued
// before any arithmetic, so each lane keeps kRowsPerGroup 16-byte loads in flight.
constexpr int kRowsPerGroup = 4;

template <int D>
// Four resident blocks per SM (<= 64 registers): more 16-byte loads in flight.
__global__ void __launch_bounds__(256, 4) k1_norm_rope_append_kernel(const __grid_constant__ K1Params p) {
    constexpr int LPR = D / 8;     // lanes per head row
    constexpr int RPW = 32 / LPR;  // row groups per warp
    constexpr int HALF = LPR / 2;  // lane distance of the rotate-half partner
    constexpr int R = kRowsPerGroup;
    const unsigned FULL = 0xffffffffu;

    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;
    const int grp = lane / LPR;
    const int H3 = p.Hq + 2 * p.Hkv;
    // A row group owns R consecutive head rows of ONE token: group g is token
    // g / RG, rows (g % RG) * R ... + R - 1 (one 32-bit division per thread).
    const int RG = (H3 + R - 1) / R;
    const int g = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * RPW + grp;
    const int t0 = g / RG;
    const int jbase = (g - t0 * RG) * R;
    const bool tok_valid = t0 < p.T;
    const int64_t t = tok_valid ? t0 : 0;
    int b = 0;
    while (b + 1 < p.nseq && t >= p.cu[b + 1]) ++b;
    const int pos = p.start[b] + static_cast<int>(t - p.cu[b]);
    const int64_t slot = static_cast<int64_t>(p.seq_slot0 + b) * p.seq_stride;

    if (blockIdx.x == 0 && threadIdx.x < p.nseq)
        p.lens[p.seq_slot0 + threadIdx.x] =
            p.start[threadIdx.x] + p.cu[threadIdx.x + 1] - p.cu[threadIdx.x];
    if (tok_valid && pos >= p.cap)  // cannot happen after host validation; never write out of bounds
        set_error(p.err, kErrBounds, kKernK1, 1);
    const bool tok_active = tok_valid && pos < p.cap;

    const uint4 wqv = __ldg(reinterpret_cast<const uint4 *>(p.wq) + sub);
    const uint4 wkv = __ldg(reinterpret_cast<const uint4 *>(p.wk) + sub);

    // Phase 1: addresses and loads of the R rows.
    uint4 xv[R];
    __nv_bfloat16 *dst[R];
    uint32_t kind[R];  // 0 = q, 1 = k, 2 = v, 3 = inactive
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int j = jbase + r;
        const bool active = tok_active && j < H3;
        const __nv_bfloat16 *src;
        if (j < p.Hq) {
            src = p.q + (t * p.Hq + j) * D;
            dst[r] = p.qp + (t * p.Hq + j) * D;
            kind[r] = 0;
        } else if (j < p.Hq + p.Hkv) {
            const int h = j - p.Hq;
            src = p.k + (t * p.Hkv + h) * D;
            dst[r] = p.kc + slot + h * p.head_stride + static_cast<int64_t>(pos) * D;
            kind[r] = 1;
        } else {
            const int h = j - p.Hq - p.Hkv;
            src = p.v + (t * p.Hkv + h) * D;
            dst[r] = p.vc + slot + h * p.head_stride + static_cast<int64_t>(pos) * D;
            kind[r] = 2;
        }
        if (!active) kind[r] = 3;
        xv[r] = active ? __ldg(reinterpret_cast<const uint4 *>(src) + sub) : make_uint4(0, 0, 0, 0);
    }
    const float4 *tab = reinterpret_cast<const float4 *>(
        p.rope + static_cast<int64_t>(tok_active ? pos : 0) * (D / 2) + 8 * (sub % HALF));
    float4 cs[4];  // (cos_a, sin_a, cos_b, sin_b) of this lane's 8 dims, shared by the R rows
#pragma unroll
    for (int e = 0; e < 4; ++e) cs[e] = __ldg(tab + e);

    // Phase 2: norm, rotate, store.
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint4 wv = kind[r] == 0 ? wqv : wkv;
        const uint32_t xw[4] = {xv[r].x, xv[r].y, xv[r].z, xv[r].w};
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
        float x[8], wf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = bf16lo(xw[e]);
            x[2 * e + 1] = bf16hi(xw[e]);
            wf[2 * e] = bf16lo(ww[e]);
            wf[2 * e + 1] = bf16hi(ww[e]);
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
        for (int o = HALF; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
        const float rr = rsqrtf(ss * (1.0f / D) + p.eps);

        // y = bf16(w * bf16(x * r)), kept packed (exact bf16 values) for the exchange.
        uint32_t yw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = wf[2 * e] * round_bf16(x[2 * e] * rr);
            const float c = wf[2 * e + 1] * round_bf16(x[2 * e + 1] * rr);
            yw[e] = pack_bf16(a, c);
        }
        uint32_t pw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pw[e] = __shfl_xor_sync(FULL, yw[e], HALF);

        const bool lower = sub < HALF;
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float y0 = bf16lo(yw[e]), y1 = bf16hi(yw[e]);
            const float q0 = bf16lo(pw[e]), q1 = bf16hi(pw[e]);
            const float r0 = lower ? y0 * cs[e].x - q0 * cs[e].y : y0 * cs[e].x + q0 * cs[e].y;
            const float r1 = lower ? y1 * cs[e].z - q1 * cs[e].w : y1 * cs[e].z + q1 * cs[e].w;
            ow[e] = pack_bf16(r0, r1);
        }
        if (kind[r] != 3) {
            const uint4 o4 = kind[r] == 2 ? xv[r] : make_uint4(ow[0], ow[1], ow[2], ow[3]);
            reinterpret_cast<uint4 *>(dst[r])[sub] = o4;
        }
    }
}

// ==================================================================== token-tiled form
// Every warp owns a two-stage ring in shared memory and walks its own share of
// the tokens (token t goes to warp t mod (CTAs x warps)).  Lane 0 copies a
// token's q, k and v rows (three contiguous runs of the packed input) into the
// next stage with bulk copies completing on the stage's mbarrier while the
// warp transforms the current stage (RMSNorm + RoPE of the q and k rows, the
// cast placement of the per-row form) and writes q', k' and v to their
// places with 16-byte stores (one row of 256 bytes per 16 lanes); the stage is
// only read, so the next copy into it follows the warp's last read of it.
// Bytes in flight: a token (12 KB at the Qwen3-4B geometry) per warp, eight
// warps per SM.
// RMSNorm + RoPE of this lane's 8 dims of a head row (lpr lanes per row, the
// rotate-half partner lpr/2 lanes away): x_hat = bf16(x * r), y = bf16(w *
// x_hat) (a bf16x2 multiply: the product of two bf16 values is exact in fp32,
// so it rounds exactly as the per-block form's fp32 multiply does), then the
// rotation in fp32 pairs and one rounding.  sn holds the sines signed for this
// lane's half (-sin below D/2, +sin above).
__device__ __forceinline__ uint4 k1_norm_rope16(uint4 xv, uint4 wv, const float2 (&cs2)[4],
                                               const float2 (&sn2)[4], float eps, int lpr) {
    const unsigned FULL = 0xffffffffu;
    const int half = lpr / 2;
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
    float2 x[4];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[e] = make_float2(bf16lo(xw[e]), bf16hi(xw[e]));
        ss = fmaf(x[e].x, x[e].x, fmaf(x[e].y, x[e].y, ss));
    }
    for (int o = half; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
    const float rr = rsqrtf(ss * (1.0f / static_cast<float>(lpr * 8)) + eps);
    const float2 r2 = make_float2(rr, rr);
    uint32_t yw[4], pw[4], ow[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 xh = __fmul2_rn(x[e], r2);
        const uint32_t xb = pack_bf16(xh.x, xh.y);
        const __nv_bfloat162 y = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&xb),
                                         *reinterpret_cast<const __nv_bfloat162 *>(&ww[e]));
        yw[e] = *reinterpret_cast<const uint32_t *>(&y);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) pw[e] = __shfl_xor_sync(FULL, yw[e], half);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 y = make_float2(bf16lo(yw[e]), bf16hi(yw[e]));
        const float2 q = make_float2(bf16lo(pw[e]), bf16hi(pw[e]));
        const float2 rot = __ffma2_rn(q, sn2[e], __fmul2_rn(y, cs2[e]));
        ow[e] = pack_bf16(rot.x, rot.y);
    }
    return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

constexpr int kK1TWarps = 8;  // warps per CTA, one CTA per SM

template <int D>
__global__ void __launch_bounds__(kK1TWarps * 32, 1)
    k1t_norm_rope_append_kernel(const __grid_constant__ K1Params p) {
    constexpr int LPR = D / 8;     // lanes per head row
    constexpr int RPW = 32 / LPR;  // rows per warp pass
    constexpr int HALF = LPR / 2;
    const unsigned FULL = 0xffffffffu;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar[kK1TWarps * 2];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane % LPR, grp = lane / LPR;
    // When the prefill attention kernel follows (launched as a programmatic
    // dependent), its set-up may start now; it reads q' and the cache only
    // after this grid has finished.
    if (p.signal_early) griddep_launch_dependents();
    const uint32_t qbytes = static_cast<uint32_t>(p.Hq) * D * 2;
    const uint32_t kvbytes = static_cast<uint32_t>(p.Hkv) * D * 2;
    const uint32_t stage_bytes = (qbytes + 2 * kvbytes + 127) & ~127u;
    uint8_t *ring = smem + static_cast<size_t>(warp) * 2 * stage_bytes;
    const uint32_t bar0 = smem_u32(&bar[2 * warp]);

    if (blockIdx.x == 0 && threadIdx.x < p.nseq)
        p.lens[p.seq_slot0 + threadIdx.x] =
            p.start[threadIdx.x] + p.cu[threadIdx.x + 1] - p.cu[threadIdx.x];
    if (lane == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint4 wqv = __ldg(reinterpret_cast<const uint4 *>(p.wq) + sub);
    const uint4 wkv = __ldg(reinterpret_cast<const uint4 *>(p.wk) + sub);

    const int64_t stride = static_cast<int64_t>(gridDim.x) * kK1TWarps;
    int64_t t = static_cast<int64_t>(blockIdx.x) * kK1TWarps + warp;
    auto load = [&](int64_t tok, int s) {  // lane 0 only
        const uint32_t dst = smem_u32(ring + s * stage_bytes);
        const uint32_t b = bar0 + 8 * s;
        mbar_expect_tx(b, qbytes + 2 * kvbytes);
        bulk_g2s(dst, p.q + tok * p.Hq * D, qbytes, b);
        bulk_g2s(dst + qbytes, p.k + tok * p.Hkv * D, kvbytes, b);
        bulk_g2s(dst + qbytes + kvbytes, p.v + tok * p.Hkv * D, kvbytes, b);
    };
    if (lane == 0 && t < p.T) load(t, 0);
    // Sequence and position of a token, and its row of the (cos, sin) table for
    // this lane's 8 dims.  The next token's row is loaded while the warp works
    // on the current one, so its latency stays off the token's path.
    auto locate = [&](int64_t tok, int &bb, int &pp) {
        int b = 0;
        while (b + 1 < p.nseq && tok >= p.cu[b + 1]) ++b;
        bb = b;
        pp = p.start[b] + static_cast<int>(tok - p.cu[b]);
    };
    auto rope_row = [&](int pp, float4 (&c)[4]) {
        const float4 *tab = reinterpret_cast<const float4 *>(
            p.rope + static_cast<int64_t>(pp < p.cap ? pp : 0) * (D / 2) + 8 * (sub % HALF));
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e] = __ldg(tab + e);
    };
    int b_cur = 0, pos_cur = 0;
    float4 rope_cur[4];
    if (t < p.T) {
        locate(t, b_cur, pos_cur);
        rope_row(pos_cur, rope_cur);
    }
    int abort_flag = 0;  // each warp gives up on its own
    int i = 0;
    bool ok = true;
    for (; t < p.T; ++i, t += stride) {
        const int s = i & 1;
        const int64_t tn = t + stride;
        if (lane == 0 && tn < p.T) load(tn, s ^ 1);  // the warp is done with that stage
        int b_nx = 0, pos_nx = 0;
        float4 rope_nx[4];
        if (tn < p.T) {
            locate(tn, b_nx, pos_nx);
            rope_row(pos_nx, rope_nx);
        }
        ok = mbar_wait(bar0 + 8 * s, (i >> 1) & 1, &abort_flag, p.err, kKernK1, 2);
        ok = __all_sync(FULL, ok);
        if (!ok) break;
        const int b = b_cur, pos = pos_cur;
        const bool in_cap = pos < p.cap;  // always, after host validation
        if (!in_cap && lane == 0) set_error(p.err, kErrBounds, kKernK1, 1);
        // (cos, sin) of this lane's 8 dims as pairs, the sines signed for its half
        float2 cs2[4], sn2[4];
        const float sgn = (sub % LPR) < HALF ? -1.f : 1.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 c4 = rope_cur[e];
            cs2[e] = make_float2(c4.x, c4.z);
            sn2[e] = make_float2(sgn * c4.y, sgn * c4.w);
        }
        uint8_t *st = ring + s * stage_bytes;
        const int64_t slot = static_cast<int64_t>(p.seq_slot0 + b) * p.seq_stride +
                             static_cast<int64_t>(pos) * D;
        // q and k rows: q' to the output rows, k' to its cache slot, 16 bytes per
        // lane straight from registers.  Four independent rows per lane at a time.
        constexpr int U = 4;
        const int nqk = p.Hq + p.Hkv;
        for (int r0 = 0; r0 < nqk; r0 += RPW * U) {  // warp-uniform
            uint4 xv[U];
            int rr[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                rr[u] = r0 + u * RPW + grp;
                const int rs = rr[u] < nqk ? rr[u] : 0;
                xv[u] = reinterpret_cast<const uint4 *>(st + static_cast<size_t>(rs) * D * 2)[sub];
            }
            uint4 o[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                o[u] = k1_norm_rope16(xv[u], rr[u] < p.Hq ? wqv : wkv, cs2, sn2, p.eps, LPR);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int r = rr[u];
                if (r < p.Hq)
                    reinterpret_cast<uint4 *>(p.qp + (t * p.Hq + r) * D)[sub] = o[u];
                else if (r < nqk && in_cap)
                    reinterpret_cast<uint4 *>(p.kc + slot + (r - p.Hq) * p.head_stride)[sub] = o[u];
            }
        }
        // v rows: copied bit-exactly from the stage to their cache slots.
        const uint8_t *vs = st + qbytes + kvbytes;
        for (int r0 = 0; r0 < p.Hkv; r0 += RPW) {
            const int r = r0 + grp;
            if (r < p.Hkv && in_cap)
                reinterpret_cast<uint4 *>(p.vc + slot + r * p.head_stride)[sub] =
                    reinterpret_cast<const uint4 *>(vs + static_cast<size_t>(r) * D * 2)[sub];
        }
        // The warp's reads of the stage come before the next bulk copy overwrites it.
        fence_proxy_async_smem();
        __syncwarp();
        b_cur = b_nx;
        pos_cur = pos_nx;
#pragma unroll
        for (int e = 0; e < 4; ++e) rope_cur[e] = rope_nx[e];
    }
    if (lane == 0) {
        // A copy requested for a token that was not reached (the loop gave up):
        // wait for it (bounded) before the shared memory goes away.
        if (!ok && t + stride < p.T) {
            int dummy = 0;
            mbar_wait(bar0 + 8 * ((i + 1) & 1), ((i + 1) >> 1) & 1, &dummy, p.err, kKernK1, 3);
        }
    }
}

// Shared memory of the token-tiled form for a geometry (0: a token does not fit).
static size_t k1t_smem_bytes(int Hq, int Hkv, int D) {
    const size_t stage = (static_cast<size_t>(Hq + 2 * Hkv) * D * 2 + 127) & ~static_cast<size_t>(127);
    const size_t bytes = static_cast<size_t>(kK1TWarps) * 2 * stage + 128;
    return bytes <= 200 * 1024 ? bytes : 0;
}

template <int D>
static cudaError_t launch_k1t(const K1Params &p, size_t smem, cudaStream_t stream) {
    static std::atomic<unsigned> configured{0u};  // devices 0..31 set up (one bit each)
    static std::atomic<int> sms_cache[32] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 32 || !((configured.load(std::memory_order_acquire) >> dev) & 1u)) {
        cudaError_t e = cudaFuncSetAttribute(k1t_norm_rope_append_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024 + 128);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (dev < 32) {
            sms_cache[dev].store(sms, std::memory_order_relaxed);
            configured.fetch_or(1u << dev, std::memory_order_release);
        }
    }
    int sms = dev < 32 ? sms_cache[dev].load(std::memory_order_relaxed) : 0;
    if (sms <= 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const int64_t need = (static_cast<int64_t>(p.T) + kK1TWarps - 1) / kK1TWarps;
    const int blocks = static_cast<int>(std::min<int64_t>(need, sms));
    k1t_norm_rope_append_kernel<D><<<blocks, kK1TWarps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_k1(const K1Params &p, int D, cudaStream_t stream) {
    if (p.T <= 0) return cudaSuccess;
    const size_t smem = k1t_smem_bytes(p.Hq, p.Hkv, D);
    if (smem > 0) return D == 128 ? launch_k1t<128>(p, smem, stream) : launch_k1t<64>(p, smem, stream);
    return launch_k1_rows(p, D, stream);
}

// Per-block form, for geometries whose token does not fit a stage.
cudaError_t launch_k1_rows(const K1Params &p, int D, cudaStream_t stream) {
    const int RG = (p.Hq + 2 * p.Hkv + kRowsPerGroup - 1) / kRowsPerGroup;
    const int64_t groups = static_cast<int64_t>(p.T) * RG;  // < 2^31: T is limited by the caller
    const int groups_per_block = (256 / 32) * (32 / (D / 8));
    const int64_t blocks = (groups + groups_per_block - 1) / groups_per_block;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    if (D == 128)
        k1_norm_rope_append_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    else
        k1_norm_rope_append_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace qa
