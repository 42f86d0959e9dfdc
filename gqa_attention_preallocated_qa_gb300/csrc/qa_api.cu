// qa_api.cu -- the C ABI declared in include/qa.h: cache object, argument
// validation, host mirror of the lengths, tensor-map creation and launch
// ordering on the caller's stream.  No fallback path exists: an unsupported
// shape or an invalid argument returns a status before anything is enqueued
// (the boundary rule of the pegainfer PR #862 review, "add SM120 FlashInfer
// GDN prefill candidate": invalid geometry fails validation instead of
// silently running something else).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "launch_order.h"
#include "qa.h"
#include "qa_internal.h"

static_assert(qa::LaunchOrder::kGuardAll == qa::kK3GuardAll, "one guard value for 'all rows'");

#define QA_API extern "C" __attribute__((visibility("default")))

using qa::K1Params;
using qa::K2Params;
using qa::K3Params;

struct qa_cache {
    qa_config cfg{};
    int device = 0;
    int num_sms = 0;
    int G = 1, HPC = 1, HG = 1;
    int64_t layer_elems = 0;   // elements of one layer's K (or V)
    __nv_bfloat16 *K = nullptr, *V = nullptr;
    int32_t *lens_dev = nullptr;
    float2 *rope = nullptr;
    uint32_t *err = nullptr;
    uint32_t *seq_cnt = nullptr;  // decode with device lengths: groups done per sequence
    std::vector<int> window;      // per layer: attention window in keys (0: full)
    int overlap = 6;              // decode launches whose clusters the split plan fits at once
    bool overlap_fixed = false;   // set by qa_cache_set_decode_overlap: no per-launch choice
    std::vector<CUtensorMap> maps;  // [layer][K, V] decode tensor maps (copied into each launch)
    std::vector<int32_t> lens_host;
    uint64_t kv_bytes = 0, scratch_bytes = 0;
    std::atomic<uint64_t> launches[QA_NUM_KERNELS];
};

namespace {

// Launch ordering of the decode kernel family (launch_order.h): one record of
// recent launches per stream, shared by every cache of the process.
qa::LaunchOrder g_order;

// Failure-detection test hook (qa_debug_arm_wait_timeout): the kernel index
// whose next launch withholds a copy (-1: none) and that launch's wait limit.
std::atomic<int> g_fault_kernel{-1};
std::atomic<uint64_t> g_fault_wait_ns{qa::kWaitTimeoutNs};

__global__ void qa_reset_kernel(int32_t *lens, int n_lens, uint32_t *seq_cnt, int n_seq) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_lens; i += gridDim.x * blockDim.x)
        lens[i] = 0;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_seq; i += gridDim.x * blockDim.x)
        seq_cnt[i] = 0;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_shape(const qa_config &c) {
    if (c.head_dim != 64 && c.head_dim != 128) return false;
    if (c.n_kv_heads <= 0 || c.n_q_heads <= 0 || c.n_q_heads % c.n_kv_heads) return false;
    const int G = c.n_q_heads / c.n_kv_heads;
    return G == 1 || G == 2 || G == 4 || G == 8;
}

void free_all(qa_cache *c) {
    cudaFree(c->K);
    cudaFree(c->V);
    cudaFree(c->lens_dev);
    cudaFree(c->rope);
    cudaFree(c->err);
    cudaFree(c->seq_cnt);
}

template <typename T>
bool dev_alloc(T **p, size_t count, uint64_t &acct) {
    const size_t bytes = std::max<size_t>(count, 1) * sizeof(T);
    if (cudaMalloc(reinterpret_cast<void **>(p), bytes) != cudaSuccess) {
        *p = nullptr;
        return false;
    }
    acct += bytes;
    return cudaMemset(*p, 0, bytes) == cudaSuccess;
}

qa_status check_layer(const qa_cache *c, int layer, int batch) {
    if (!c) return QA_ERR_INVALID_ARG;
    if (layer < 0 || layer >= c->cfg.num_layers) return QA_ERR_INVALID_ARG;
    if (batch < 1 || batch > c->cfg.max_batch) return QA_ERR_INVALID_ARG;
    return QA_OK;
}

// Per-sequence K (or V) tensor map over one layer's cache: (D, L, Hkv) with the
// head stride of the cache, 64 x box_rows x 1 boxes, 128-byte swizzle; rows at
// or beyond L read as zero.  K uses 64-row boxes (the CTA-pair prefill loads
// half a key tile per CTA), V 128-row boxes.
bool encode_kv_map(CUtensorMap *m, void *base, int D, int L, int Hkv, int cap, int box_rows) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                                static_cast<cuuint64_t>(Hkv)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(cap) * D * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Query tensor map over q' rows: (D, Hq, T) with 64 x 1 x 128 boxes.
bool encode_q_map(CUtensorMap *m, void *base, int D, int Hq, int T) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                                static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(Hq) * D * 2};
    const cuuint32_t box[3] = {64, 1, 128};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

qa::FaultPlan qa::take_fault(int kernel) {
    FaultPlan f;
    int armed = kernel;
    if (g_fault_kernel.load(std::memory_order_acquire) == kernel &&
        g_fault_kernel.compare_exchange_strong(armed, -1, std::memory_order_acq_rel)) {
        f.fault = 1;
        f.wait_ns = g_fault_wait_ns.load(std::memory_order_acquire);
    }
    return f;
}

bool qa::encode_decode_map(CUtensorMap *m, void *base, int D, int capacity, int rows_z) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(capacity),
                                static_cast<cuuint64_t>(rows_z)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(capacity) * D * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(qa::kK3Chunk), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// The launches a host-position decode launch plans room for (unless the caller
// fixed the number with qa_cache_set_decode_overlap): one when nothing may still
// run beside it, two when launches on its own layer may (a single-layer loop:
// the rows they append are read only after the wait, so fewer launches overlap
// usefully), and the cache's setting when only other layers' launches may (a
// loop over layers).
int plan_overlap(const qa_cache *c, cudaStream_t stream, int layer, int64_t resident_max) {
    if (c->overlap_fixed) return c->overlap;
    switch (g_order.in_flight(stream, c, layer, resident_max)) {
        case 0: return 1;
        case 2: return std::min(2, c->overlap);
        default: return c->overlap;
    }
}

// Split count for `overlap` launches of `groups` clusters.  Unless the caller
// fixed the number of launches, fewer are planned for as long as the plan
// would leave fewer than two splits (one split streams a whole sequence's
// cache per CTA, whose latency then outweighs the extra overlap).
int plan_splits(const qa_cache *c, int groups, int pos_max, bool multi, int HPC, int overlap) {
    int S = qa::k3_choose_splits(c->cfg.head_dim, HPC, groups, pos_max, multi, overlap);
    if (!c->overlap_fixed)
        for (int n = overlap - 1; S < 2 && n >= 1; --n)
            S = qa::k3_choose_splits(c->cfg.head_dim, HPC, groups, pos_max, multi, n);
    return S;
}

// overlap: launches whose clusters should fit at once (see qa_cache_set_decode_overlap).
int choose_splits(const qa_cache *c, int batch, int pos_max, int overlap) {
    return plan_splits(c, batch * c->cfg.n_kv_heads * c->HG, pos_max, false, c->HPC, overlap);
}

// Validation shared by qa_prefill and qa_prefill_transform.
qa_status check_prefill(const qa_cache *c, int layer, int batch, const int32_t *prompt_lens,
                        const void *q, const void *k, const void *v, const void *wq,
                        const void *wk, const void *dst, int64_t *T_out) {
    qa_status st = check_layer(c, layer, batch);
    if (st != QA_OK) return st;
    if (!prompt_lens) return QA_ERR_INVALID_ARG;
    // The new tokens of sequence b take positions len_b .. len_b + prompt_lens[b] - 1
    // after what the layer already holds (a chunked prefill appends).
    const int32_t *cur = c->lens_host.data() + static_cast<size_t>(layer) * c->cfg.max_batch;
    int64_t T = 0;
    for (int b = 0; b < batch; ++b) {
        if (prompt_lens[b] < 0) return QA_ERR_INVALID_ARG;
        if (static_cast<int64_t>(cur[b]) + prompt_lens[b] > c->cfg.capacity) return QA_ERR_CAPACITY;
        T += prompt_lens[b];
    }
    if (T > 0) {
        if (!q || !k || !v || !wq || !wk || !dst) return QA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(wq) || !aligned16(wk) ||
            !aligned16(dst))
            return QA_ERR_ALIGNMENT;
        if (T > (int64_t(1) << 26)) return QA_ERR_INVALID_ARG;  // keeps K1's 32-bit row-group index
    }
    *T_out = T;
    return QA_OK;
}

K1Params make_k1(qa_cache *c, int layer, const void *q, const void *k, const void *v,
                 const void *wq, const void *wk, void *qp) {
    const qa_config &g = c->cfg;
    K1Params p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.wq = static_cast<const __nv_bfloat16 *>(wq);
    p.wk = static_cast<const __nv_bfloat16 *>(wk);
    p.qp = static_cast<__nv_bfloat16 *>(qp);
    p.kc = c->K + layer * c->layer_elems;
    p.vc = c->V + layer * c->layer_elems;
    p.lens = c->lens_dev + static_cast<int64_t>(layer) * g.max_batch;
    p.rope = c->rope;
    p.err = c->err;
    p.head_stride = static_cast<int64_t>(g.capacity) * g.head_dim;
    p.seq_stride = p.head_stride * g.n_kv_heads;
    p.Hq = g.n_q_heads;
    p.Hkv = g.n_kv_heads;
    p.cap = g.capacity;
    p.eps = g.rms_eps;
    return p;
}

// K1 over all prompt rows, in launches of up to kMaxSeqPerLaunch sequences.
// then_k2: the prefill attention launches follow at once on the stream; K1
// then lets them start their set-up early (programmatic dependent launch).
qa_status run_k1(qa_cache *c, int layer, int batch, const int32_t *lens, const void *q,
                 const void *k, const void *v, const void *wq, const void *wk, void *qp,
                 cudaStream_t s, bool then_k2) {
    const qa_config &g = c->cfg;
    const int D = g.head_dim;
    int64_t row0 = 0;
    for (int s0 = 0; s0 < batch; s0 += qa::kMaxSeqPerLaunch) {
        const int n = std::min(qa::kMaxSeqPerLaunch, batch - s0);
        K1Params p = make_k1(c, layer, static_cast<const __nv_bfloat16 *>(q) + row0 * g.n_q_heads * D,
                             static_cast<const __nv_bfloat16 *>(k) + row0 * g.n_kv_heads * D,
                             static_cast<const __nv_bfloat16 *>(v) + row0 * g.n_kv_heads * D, wq,
                             wk, static_cast<__nv_bfloat16 *>(qp) + row0 * g.n_q_heads * D);
        p.nseq = n;
        p.seq_slot0 = s0;
        p.cu[0] = 0;
        const int32_t *cur = c->lens_host.data() + static_cast<size_t>(layer) * g.max_batch;
        for (int i = 0; i < n; ++i) {
            p.cu[i + 1] = p.cu[i] + lens[s0 + i];
            p.start[i] = cur[s0 + i];
        }
        p.T = p.cu[n];
        p.signal_early = then_k2 ? 1 : 0;
        if (p.T > 0) {
            if (qa::launch_k1(p, D, s) != cudaSuccess) return QA_ERR_CUDA;
            g_order.barrier(s);
            c->launches[QA_KERNEL_NORM_ROPE_APPEND]++;
        }
        row0 += p.T;
    }
    return QA_OK;
}

// The decode kernel's parameters common to every launch on `layer`.
K3Params make_k3(qa_cache *c, int layer, const void *q, const void *k, const void *v,
                 const void *wq, const void *wk, void *out) {
    const qa_config &g = c->cfg;
    K3Params p{};
    p.tmk = c->maps[2 * layer];
    p.tmv = c->maps[2 * layer + 1];
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.wq = static_cast<const __nv_bfloat16 *>(wq);
    p.wk = static_cast<const __nv_bfloat16 *>(wk);
    p.kc = c->K + layer * c->layer_elems;
    p.vc = c->V + layer * c->layer_elems;
    p.lens = c->lens_dev + static_cast<int64_t>(layer) * g.max_batch;
    p.rope = c->rope;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.err = c->err;
    p.head_stride = static_cast<int64_t>(g.capacity) * g.head_dim;
    p.seq_stride = p.head_stride * g.n_kv_heads;
    p.Hq = g.n_q_heads;
    p.Hkv = g.n_kv_heads;
    p.G = c->G;
    p.HG = c->HG;
    p.cap = g.capacity;
    p.eps = g.rms_eps;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(g.head_dim)));
    p.seq_cnt = c->seq_cnt;
    p.window = c->window[layer];
    p.fault = 0;
    p.wait_ns = qa::kWaitTimeoutNs;
    return p;
}

// A chunk of at most kK3MaxTokens new tokens per sequence (a verify step, a
// short append) runs as multi-token launches of the decode kernel, one per 64
// sequences that have new tokens: every (sequence, kv head) streams its cache
// once for all of its new tokens.  A CTA holds HPC heads x 8 / HPC tokens.
qa_status run_multi(qa_cache *c, int layer, int batch, const int32_t *lens, int tmax,
                    const void *q, const void *k, const void *v, const void *wq, const void *wk,
                    void *out, cudaStream_t s) {
    const qa_config &g = c->cfg;
    int HPC = c->HPC;
    while (HPC > 1 && qa::kK3MaxTokens / HPC < tmax) HPC /= 2;
    K3Params p = make_k3(c, layer, q, k, v, wq, wk, out);
    p.HG = c->G / HPC;
    const int32_t *mirror = c->lens_host.data() + static_cast<size_t>(layer) * g.max_batch;
    std::vector<std::pair<K3Params, qa::K3Multi>> launches;
    qa::K3Multi m{};
    int nz = 0, row = 0, pos_max = 0;
    const int resident_max = qa::k3_max_resident_ctas();
    const int ov = plan_overlap(c, s, layer, resident_max);
    auto flush = [&]() {
        if (nz == 0) return;
        p.B = nz;
        p.S = plan_splits(c, nz * g.n_kv_heads * p.HG, pos_max, true, HPC,
                          launches.empty() ? ov : std::min(2, ov));
        launches.emplace_back(p, m);
        nz = 0;
        pos_max = 0;
    };
    for (int b = 0; b < batch; ++b) {
        if (lens[b] > 0) {
            m.seq[nz] = b;
            m.ntok[nz] = lens[b];
            m.row0[nz] = row;
            p.pos[nz] = mirror[b];
            pos_max = std::max(pos_max, static_cast<int>(mirror[b]));
            if (++nz == qa::kK3MaxSeqPerLaunch) flush();
        }
        row += lens[b];
    }
    flush();
    for (auto &l : launches) {
        int tm = 0;
        for (int z = 0; z < l.first.B; ++z) tm = std::max(tm, l.second.ntok[z]);
        l.first.guard = g_order.admit(s, c, layer, l.first.S * g.n_kv_heads * l.first.HG * l.first.B,
                                      tm, true, resident_max);
        const qa::FaultPlan f = qa::take_fault(QA_KERNEL_DECODE_ATTN);
        l.first.fault = f.fault;
        l.first.wait_ns = f.wait_ns;
        if (qa::launch_k3_multi(l.first, l.second, g.head_dim, HPC, s) != cudaSuccess) {
            // The launches before this one were enqueued and advance their
            // sequences' device lengths: the host copy follows them.
            int32_t *host = c->lens_host.data() + static_cast<size_t>(layer) * g.max_batch;
            for (auto *e = launches.data(); e != &l; ++e)
                for (int z = 0; z < e->first.B; ++z) host[e->second.seq[z]] += e->second.ntok[z];
            return QA_ERR_CUDA;
        }
        c->launches[QA_KERNEL_DECODE_ATTN]++;
    }
    return QA_OK;
}

// One prefill-attention launch (up to kMaxSeqPerLaunch sequences) and its work items.
struct PrefillLaunch {
    K2Params p;
    int items;
};

// K2 launches for the L_b = lens[b] new tokens of each sequence, at positions
// start[b] .. start[b] + L_b - 1 of `layer` (already in the cache when the
// launches run); q' rows are read from `qprime` and the outputs written to
// `out` (both packed [T][Hq][D]; they may be the same buffer).  Builds every
// tensor map first, so a failure leaves nothing enqueued.
qa_status plan_k2(qa_cache *c, int layer, int batch, const int32_t *lens, const int32_t *start,
                  const void *qprime, void *out, std::vector<PrefillLaunch> &launches) {
    const qa_config &g = c->cfg;
    const int D = g.head_dim;
    int64_t row0 = 0;
    for (int s0 = 0; s0 < batch; s0 += qa::kMaxSeqPerLaunch) {
        const int n = std::min(qa::kMaxSeqPerLaunch, batch - s0);
        K2Params p{};
        int nseq = 0, rows = 0, maxqb = 0;
        for (int i = 0; i < n; ++i) {
            const int L = lens[s0 + i];
            const int P = start[s0 + i];
            if (L > 0) {
                __nv_bfloat16 *kb = c->K + layer * c->layer_elems +
                                    static_cast<int64_t>(s0 + i) * g.n_kv_heads * g.capacity * D;
                __nv_bfloat16 *vb = c->V + layer * c->layer_elems +
                                    static_cast<int64_t>(s0 + i) * g.n_kv_heads * g.capacity * D;
                if (!encode_kv_map(&p.tm_k[nseq], kb, D, P + L, g.n_kv_heads, g.capacity, 64) ||
                    !encode_kv_map(&p.tm_v[nseq], vb, D, P + L, g.n_kv_heads, g.capacity, 128))
                    return QA_ERR_CUDA;
                p.len[nseq] = L;
                p.start[nseq] = P;
                p.cu[nseq] = rows;
                maxqb = std::max(maxqb, (L + 127) / 128);
                ++nseq;
            }
            rows += L;
        }
        if (nseq > 0) {
            if (!encode_q_map(&p.tm_q,
                              const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(qprime)) +
                                  row0 * g.n_q_heads * D,
                              D, g.n_q_heads, rows))
                return QA_ERR_CUDA;
            p.out = static_cast<__nv_bfloat16 *>(out) + row0 * g.n_q_heads * D;
            p.err = c->err;
            p.nseq = nseq;
            p.Hq = g.n_q_heads;
            p.Hkv = g.n_kv_heads;
            p.G = c->G;
            p.npairs = (c->G + 1) / 2;  // two-head items; the launch may halve them
            p.max_qblocks = maxqb;
            p.window = c->window[layer];
            p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
            p.fault = 0;
            p.wait_ns = qa::kWaitTimeoutNs;
            int items = 0;
            for (int i = 0; i < nseq; ++i) items += (p.len[i] + 127) / 128;
            items *= g.n_kv_heads * p.npairs;
            launches.push_back({p, items});
        }
        row0 += rows;
    }
    return QA_OK;
}

qa_status launch_k2s(qa_cache *c, std::vector<PrefillLaunch> &launches, cudaStream_t s) {
    for (auto &l : launches) {
        const qa::FaultPlan f = qa::take_fault(QA_KERNEL_PREFILL_ATTN);
        l.p.fault = f.fault;
        l.p.wait_ns = f.wait_ns;
        if (qa::launch_k2(l.p, c->cfg.head_dim, l.items, s) != cudaSuccess) return QA_ERR_CUDA;
        g_order.barrier(s);
        c->launches[QA_KERNEL_PREFILL_ATTN]++;
    }
    return QA_OK;
}

}  // namespace

// ============================================================== public API

QA_API int qa_abi_version(void) { return QA_ABI_VERSION; }

QA_API const char *qa_status_str(qa_status s) {
    switch (s) {
        case QA_OK: return "ok";
        case QA_ERR_INVALID_ARG: return "invalid argument";
        case QA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case QA_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
        case QA_ERR_CAPACITY: return "cache capacity exceeded";
        case QA_ERR_STATE: return "invalid cache state";
        case QA_ERR_CUDA: return "CUDA runtime error";
        case QA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case QA_ERR_DEVICE_BOUNDS: return "device position out of bounds";
    }
    return "unknown status";
}

QA_API qa_status qa_cache_alloc(const qa_config *cfg, qa_cache **out) {
    if (!cfg || !out) return QA_ERR_INVALID_ARG;
    *out = nullptr;
    const qa_config g = *cfg;
    if (g.num_layers <= 0 || g.max_batch <= 0 || g.capacity <= 0 || g.n_q_heads <= 0 ||
        g.n_kv_heads <= 0 || g.head_dim <= 0 || !(g.rope_theta > 0.f) || !(g.rms_eps >= 0.f))
        return QA_ERR_INVALID_ARG;
    if (!supported_shape(g)) return QA_ERR_UNSUPPORTED_SHAPE;
    if (g.capacity > (1 << 24) || g.max_batch > 65535) return QA_ERR_UNSUPPORTED_SHAPE;

    qa_cache *c = new (std::nothrow) qa_cache();
    if (!c) return QA_ERR_CUDA;
    c->cfg = g;
    for (auto &x : c->launches) x = 0;
    c->G = g.n_q_heads / g.n_kv_heads;
    c->HPC = std::min(c->G, 4);
    c->HG = c->G / c->HPC;
    if (cudaGetDevice(&c->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) !=
            cudaSuccess) {
        delete c;
        return QA_ERR_CUDA;
    }
    const int D = g.head_dim;
    c->layer_elems = static_cast<int64_t>(g.max_batch) * g.n_kv_heads * g.capacity * D;
    const size_t kv = static_cast<size_t>(c->layer_elems) * g.num_layers;
    uint64_t kvb = 0, scr = 0;
    bool ok = dev_alloc(&c->K, kv, kvb) && dev_alloc(&c->V, kv, kvb) &&
              dev_alloc(&c->lens_dev, static_cast<size_t>(g.num_layers) * g.max_batch, scr) &&
              dev_alloc(&c->rope, static_cast<size_t>(g.capacity) * (D / 2), scr) &&
              dev_alloc(&c->err, 1, scr) &&
              dev_alloc(&c->seq_cnt, static_cast<size_t>(g.max_batch), scr);
    if (ok) {
        // Rotary table in fp64, stored as fp32 (cos, sin): angle = pos * theta^(-2i/D).
        std::vector<float2> tab(static_cast<size_t>(g.capacity) * (D / 2));
        for (int pos = 0; pos < g.capacity; ++pos)
            for (int i = 0; i < D / 2; ++i) {
                const double a = static_cast<double>(pos) *
                                 std::pow(static_cast<double>(g.rope_theta), -2.0 * i / D);
                tab[static_cast<size_t>(pos) * (D / 2) + i] =
                    make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
            }
        ok = cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) ==
                 cudaSuccess;
    }
    if (ok) {
        // Decode tensor maps, two per layer, kept on the host and copied into the
        // parameters of every decode launch.
        std::vector<CUtensorMap> maps(static_cast<size_t>(2) * g.num_layers);
        for (int l = 0; ok && l < g.num_layers; ++l)
            ok = qa::encode_decode_map(&maps[2 * l], c->K + l * c->layer_elems, D, g.capacity,
                                       g.max_batch * g.n_kv_heads) &&
                 qa::encode_decode_map(&maps[2 * l + 1], c->V + l * c->layer_elems, D, g.capacity,
                                       g.max_batch * g.n_kv_heads);
        ok = ok && cudaDeviceSynchronize() == cudaSuccess;
        if (ok) c->maps = std::move(maps);
    }
    if (!ok) {
        free_all(c);
        delete c;
        cudaGetLastError();
        return QA_ERR_CUDA;
    }
    c->lens_host.assign(static_cast<size_t>(g.num_layers) * g.max_batch, 0);
    c->window.assign(static_cast<size_t>(g.num_layers), 0);
    c->kv_bytes = kvb;
    c->scratch_bytes = scr;
    *out = c;
    return QA_OK;
}

QA_API qa_status qa_cache_free(qa_cache *c) {
    if (!c) return QA_OK;
    cudaDeviceSynchronize();
    g_order.clear();
    free_all(c);
    delete c;
    return QA_OK;
}

QA_API qa_status qa_cache_reset(qa_cache *c, void *stream) {
    if (!c) return QA_ERR_INVALID_ARG;
    const qa_config &g = c->cfg;
    const int n_lens = g.num_layers * g.max_batch;
    qa_reset_kernel<<<1, 256, 0, static_cast<cudaStream_t>(stream)>>>(c->lens_dev, n_lens,
                                                                       c->seq_cnt, g.max_batch);
    if (cudaGetLastError() != cudaSuccess) return QA_ERR_CUDA;
    g_order.barrier(static_cast<cudaStream_t>(stream));
    c->launches[QA_KERNEL_RESET]++;
    std::fill(c->lens_host.begin(), c->lens_host.end(), 0);
    return QA_OK;
}

QA_API qa_status qa_prefill_transform(qa_cache *c, int layer, int batch,
                                      const int32_t *prompt_lens, const void *q, const void *k,
                                      const void *v, const void *q_norm_w, const void *k_norm_w,
                                      void *qprime_out, void *stream) {
    int64_t T = 0;
    qa_status st = check_prefill(c, layer, batch, prompt_lens, q, k, v, q_norm_w, k_norm_w,
                                 qprime_out, &T);
    if (st != QA_OK) return st;
    st = run_k1(c, layer, batch, prompt_lens, q, k, v, q_norm_w, k_norm_w, qprime_out,
                static_cast<cudaStream_t>(stream), false);
    if (st != QA_OK) return st;
    for (int b = 0; b < batch; ++b)
        c->lens_host[static_cast<size_t>(layer) * c->cfg.max_batch + b] += prompt_lens[b];
    return QA_OK;
}

QA_API qa_status qa_prefill(qa_cache *c, int layer, int batch, const int32_t *prompt_lens,
                            const void *q, const void *k, const void *v, const void *q_norm_w,
                            const void *k_norm_w, void *out, void *stream) {
    int64_t T = 0;
    qa_status st =
        check_prefill(c, layer, batch, prompt_lens, q, k, v, q_norm_w, k_norm_w, out, &T);
    if (st != QA_OK) return st;
    const qa_config &g = c->cfg;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int tmax = 0;
    for (int b = 0; b < batch; ++b) tmax = std::max(tmax, static_cast<int>(prompt_lens[b]));
    if (tmax > 0 && tmax <= qa::kK3MaxTokens) {
        st = run_multi(c, layer, batch, prompt_lens, tmax, q, k, v, q_norm_w, k_norm_w, out, s);
        if (st != QA_OK) return st;
        for (int b = 0; b < batch; ++b)
            c->lens_host[static_cast<size_t>(layer) * g.max_batch + b] += prompt_lens[b];
        return QA_OK;
    }
    // Build all tensor maps before the first launch so a failure enqueues nothing.
    std::vector<PrefillLaunch> k2s;
    const int32_t *cur = c->lens_host.data() + static_cast<size_t>(layer) * g.max_batch;
    st = plan_k2(c, layer, batch, prompt_lens, cur, out, out, k2s);
    if (st != QA_OK) return st;
    // K1 stages the normed, rotated queries in `out`; K2 reads them back and
    // overwrites every row with its attention output (each CTA owns its rows).
    st = run_k1(c, layer, batch, prompt_lens, q, k, v, q_norm_w, k_norm_w, out, s, true);
    if (st != QA_OK) return st;
    st = launch_k2s(c, k2s, s);
    if (st != QA_OK) {
        // A K1 launch that signalled early is no longer followed by a kernel
        // that waits for it: let it finish before anything else is enqueued.
        cudaStreamSynchronize(s);
        return st;
    }
    for (int b = 0; b < batch; ++b)
        c->lens_host[static_cast<size_t>(layer) * g.max_batch + b] += prompt_lens[b];
    return QA_OK;
}

QA_API qa_status qa_prefill_attend(qa_cache *c, int layer, int batch, const int32_t *prompt_lens,
                                   const void *qprime, void *out, void *stream) {
    qa_status st = check_layer(c, layer, batch);
    if (st != QA_OK) return st;
    if (!prompt_lens) return QA_ERR_INVALID_ARG;
    const qa_config &g = c->cfg;
    // The new tokens are the last prompt_lens[b] positions sequence b holds.
    const int32_t *held = c->lens_host.data() + static_cast<size_t>(layer) * g.max_batch;
    std::vector<int32_t> start(static_cast<size_t>(batch));
    int64_t T = 0;
    for (int b = 0; b < batch; ++b) {
        if (prompt_lens[b] < 0 || prompt_lens[b] > held[b]) return QA_ERR_INVALID_ARG;
        start[b] = held[b] - prompt_lens[b];
        T += prompt_lens[b];
    }
    if (T == 0) return QA_OK;
    if (!qprime || !out) return QA_ERR_INVALID_ARG;
    if (!aligned16(qprime) || !aligned16(out)) return QA_ERR_ALIGNMENT;
    if (T > (int64_t(1) << 26)) return QA_ERR_INVALID_ARG;
    std::vector<PrefillLaunch> k2s;
    st = plan_k2(c, layer, batch, prompt_lens, start.data(), qprime, out, k2s);
    if (st != QA_OK) return st;
    return launch_k2s(c, k2s, static_cast<cudaStream_t>(stream));
}

QA_API int qa_decode_splits(qa_cache *c, int layer, int batch) {
    if (check_layer(c, layer, batch) != QA_OK) return 0;
    batch = std::min(batch, qa::kK3MaxSeqPerLaunch);  // the first launch of the step
    int pos_max = 0;
    for (int b = 0; b < batch; ++b)
        pos_max = std::max(pos_max, c->lens_host[static_cast<size_t>(layer) * c->cfg.max_batch + b]);
    return choose_splits(c, batch, pos_max, c->overlap);
}

namespace {
// One decode step of `layer` for sequences 0..batch-1, one launch per 64 of
// them.  dev_pos = false: positions from the host copy of the lengths (checked
// against the capacity here), which advances; true: the kernel reads and
// advances the device lengths and checks the capacity itself.
qa_status decode_step(qa_cache *c, int layer, int batch, const void *q, const void *k,
                      const void *v, const void *q_norm_w, const void *k_norm_w, void *out,
                      void *stream, bool dev_pos) {
    qa_status st = check_layer(c, layer, batch);
    if (st != QA_OK) return st;
    if (!q || !k || !v || !q_norm_w || !k_norm_w || !out) return QA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_norm_w) ||
        !aligned16(k_norm_w) || !aligned16(out))
        return QA_ERR_ALIGNMENT;
    const qa_config &g = c->cfg;
    // The host copy of the lengths is exact while every change goes through
    // this library, so host positions travel in the launch parameters and the
    // kernel never waits on reading them; the kernel still sets the device
    // lengths.  With device lengths the host copy only sizes the split plan.
    int32_t *mirror = c->lens_host.data() + static_cast<size_t>(layer) * g.max_batch;
    if (!dev_pos)
        for (int b = 0; b < batch; ++b)
            if (mirror[b] + 1 > g.capacity) return QA_ERR_CAPACITY;
    K3Params p = make_k3(c, layer, q, k, v, q_norm_w, k_norm_w, out);
    const int64_t resident_max = qa::k3_max_resident_ctas();
    // Device positions: when no launch that may still be running writes this
    // layer (a multi-layer loop, e.g. a captured layer stack), the kernel reads
    // them at once and overlaps its predecessor like a host-position step;
    // otherwise it waits for its predecessor before reading them and nothing
    // overlaps.
    const bool settled =
        dev_pos && g_order.layer_settled(static_cast<cudaStream_t>(stream), c, layer, resident_max);
    p.dev_pos = dev_pos ? (settled ? 2 : 1) : 0;
    for (int b0 = 0; b0 < batch; b0 += qa::kK3MaxSeqPerLaunch) {
        const int nb = std::min(qa::kK3MaxSeqPerLaunch, batch - b0);
        int pos_max = 0;
        for (int i = 0; i < nb; ++i) {
            p.pos[i] = mirror[b0 + i];
            pos_max = std::max(pos_max, mirror[b0 + i]);
        }
        // The host copy lags behind device positions (a captured step runs at
        // every later position): plan the splits for a full cache.
        if (dev_pos) pos_max = g.capacity - 1;
        p.b0 = b0;
        p.B = nb;
        // Device positions: the cache's overlap setting alone sets the plan (not
        // what runs beside the launch), so a captured step and the same step run
        // eagerly agree bit for bit.  Host positions: the plan follows the stream.
        p.S = choose_splits(c, nb, pos_max,
                            dev_pos ? c->overlap
                                    : plan_overlap(c, static_cast<cudaStream_t>(stream), layer,
                                                   resident_max));
        p.guard = g_order.admit(static_cast<cudaStream_t>(stream), c, layer,
                                p.S * g.n_kv_heads * c->HG * nb, 1, !dev_pos || settled,
                                resident_max);
        const qa::FaultPlan f = qa::take_fault(QA_KERNEL_DECODE_ATTN);
        p.fault = f.fault;
        p.wait_ns = f.wait_ns;
        if (qa::launch_k3(p, g.head_dim, c->HPC, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
            // The launches before this one were enqueued and advance their
            // sequences' device lengths: the host copy follows them.
            if (!dev_pos)
                for (int b = 0; b < b0; ++b) mirror[b] += 1;
            return QA_ERR_CUDA;
        }
        c->launches[QA_KERNEL_DECODE_ATTN]++;
    }
    if (!dev_pos)
        for (int b = 0; b < batch; ++b) mirror[b] += 1;
    return QA_OK;
}
}  // namespace

QA_API qa_status qa_decode_step(qa_cache *c, int layer, int batch, const void *q, const void *k,
                                const void *v, const void *q_norm_w, const void *k_norm_w,
                                void *out, void *stream) {
    return decode_step(c, layer, batch, q, k, v, q_norm_w, k_norm_w, out, stream, false);
}

QA_API qa_status qa_decode_step_device_lengths(qa_cache *c, int layer, int batch, const void *q,
                                               const void *k, const void *v, const void *q_norm_w,
                                               const void *k_norm_w, void *out, void *stream) {
    return decode_step(c, layer, batch, q, k, v, q_norm_w, k_norm_w, out, stream, true);
}

QA_API qa_status qa_cache_set_decode_overlap(qa_cache *c, int launches) {
    if (!c || launches < 1 || launches > 8) return QA_ERR_INVALID_ARG;
    c->overlap = launches;
    c->overlap_fixed = true;
    return QA_OK;
}

QA_API qa_status qa_cache_set_window(qa_cache *c, int layer, int window) {
    if (!c || layer < 0 || layer >= c->cfg.num_layers || window < 0) return QA_ERR_INVALID_ARG;
    c->window[layer] = window;
    return QA_OK;
}

QA_API qa_status qa_cache_sync_lengths(qa_cache *c, int layer, void *stream) {
    if (!c || layer < 0 || layer >= c->cfg.num_layers) return QA_ERR_INVALID_ARG;
    const qa_config &g = c->cfg;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(c->lens_host.data() + static_cast<size_t>(layer) * g.max_batch,
                        c->lens_dev + static_cast<int64_t>(layer) * g.max_batch,
                        sizeof(int32_t) * g.max_batch, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return QA_ERR_CUDA;
    g_order.barrier(s);
    return QA_OK;
}

QA_API qa_status qa_cache_view(qa_cache *c, int layer, void **k, void **v, int32_t **lens,
                               int64_t strides[4]) {
    if (!c || layer < 0 || layer >= c->cfg.num_layers) return QA_ERR_INVALID_ARG;
    const qa_config &g = c->cfg;
    if (k) *k = c->K + layer * c->layer_elems;
    if (v) *v = c->V + layer * c->layer_elems;
    if (lens) *lens = c->lens_dev + static_cast<int64_t>(layer) * g.max_batch;
    if (strides) {
        strides[3] = 1;
        strides[2] = g.head_dim;
        strides[1] = static_cast<int64_t>(g.capacity) * g.head_dim;
        strides[0] = strides[1] * g.n_kv_heads;
    }
    return QA_OK;
}

QA_API qa_status qa_cache_set_lengths(qa_cache *c, int layer, const int32_t *lens_host,
                                      void *stream) {
    if (!c || !lens_host || layer < 0 || layer >= c->cfg.num_layers) return QA_ERR_INVALID_ARG;
    const qa_config &g = c->cfg;
    for (int b = 0; b < g.max_batch; ++b)
        if (lens_host[b] < 0 || lens_host[b] > g.capacity) return QA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(c->lens_dev + static_cast<int64_t>(layer) * g.max_batch, lens_host,
                        sizeof(int32_t) * g.max_batch, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return QA_ERR_CUDA;
    g_order.barrier(s);
    std::copy(lens_host, lens_host + g.max_batch,
              c->lens_host.begin() + static_cast<size_t>(layer) * g.max_batch);
    return QA_OK;
}

QA_API qa_status qa_cache_lengths(qa_cache *c, int layer, int32_t *lens_host) {
    if (!c || !lens_host || layer < 0 || layer >= c->cfg.num_layers) return QA_ERR_INVALID_ARG;
    std::copy(c->lens_host.begin() + static_cast<size_t>(layer) * c->cfg.max_batch,
              c->lens_host.begin() + static_cast<size_t>(layer + 1) * c->cfg.max_batch, lens_host);
    return QA_OK;
}

QA_API qa_status qa_get_device_error(qa_cache *c, uint32_t *detail) {
    if (!c) return QA_ERR_INVALID_ARG;
    uint32_t word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, c->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(c->err, 0, sizeof(word)) != cudaSuccess)
        return QA_ERR_CUDA;
    g_order.clear();
    if (detail) *detail = word;
    switch (word & 0xffu) {
        case 0: return QA_OK;
        case qa::kErrTimeout: return QA_ERR_DEVICE_TIMEOUT;
        default: return QA_ERR_DEVICE_BOUNDS;
    }
}

QA_API qa_status qa_debug_arm_wait_timeout(int kernel, uint32_t wait_us) {
    if (kernel == -1) {
        g_fault_kernel.store(-1, std::memory_order_release);
        return QA_OK;
    }
    if (kernel != QA_KERNEL_PREFILL_ATTN && kernel != QA_KERNEL_DECODE_ATTN) return QA_ERR_INVALID_ARG;
    if (wait_us < 1 || wait_us > 2000000) return QA_ERR_INVALID_ARG;
    g_fault_wait_ns.store(static_cast<uint64_t>(wait_us) * 1000ull, std::memory_order_release);
    g_fault_kernel.store(kernel, std::memory_order_release);
    return QA_OK;
}

QA_API qa_status qa_stats(qa_cache *c, uint64_t launches[QA_NUM_KERNELS]) {
    if (!c || !launches) return QA_ERR_INVALID_ARG;
    for (int i = 0; i < QA_NUM_KERNELS; ++i) launches[i] = c->launches[i].load();
    return QA_OK;
}

QA_API qa_status qa_memory_info(qa_cache *c, uint64_t *kv_bytes, uint64_t *scratch_bytes) {
    if (!c) return QA_ERR_INVALID_ARG;
    if (kv_bytes) *kv_bytes = c->kv_bytes;
    if (scratch_bytes) *scratch_bytes = c->scratch_bytes;
    return QA_OK;
}
