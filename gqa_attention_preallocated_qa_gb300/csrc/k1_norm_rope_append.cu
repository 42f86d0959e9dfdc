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
#include "qa_device.cuh"

namespace qa {

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

cudaError_t launch_k1(const K1Params &p, int D, cudaStream_t stream) {
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
