// qa_internal.h -- definitions shared by the host launchers and the kernels
// (parameter blocks, limits, error kinds).  Not part of the public ABI.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through the runtime)
#include <cuda_bf16.h>
#include <stdint.h>

namespace qa {

// Error word layout: kind | kernel << 8 | site << 16.
constexpr uint32_t kErrTimeout = 1;
constexpr uint32_t kErrBounds = 2;
constexpr uint32_t kKernK1 = 1, kKernK2 = 2, kKernK3 = 3;

// Every spin on an mbarrier gives up after this long (a normal launch of any
// kernel here takes well under a millisecond).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Failure-detection test hook (qa_debug_arm_wait_timeout): a launch whose
// `fault` field is set withholds one tile copy (prefill: V tile 0 of its first
// thread block; decode: the first cache chunk of every block of the first
// cluster that streams any), so a consumer of that tile waits for an mbarrier
// no copy will ever complete, and the launch's waits give up after `wait_ns`.
// Nothing else changes.
struct FaultPlan {
    uint64_t wait_ns = kWaitTimeoutNs;
    int fault = 0;
};
// Takes (and disarms) the armed fault for `kernel` (QA_KERNEL_* index), if any.
FaultPlan take_fault(int kernel);

// ---------------------------------------------------------------- K1
// Sequences per prefill launch (K1 and K2 take their per-sequence data as
// kernel parameters; longer batches are split into several launches).
constexpr int kMaxSeqPerLaunch = 8;

struct K1Params {
    const __nv_bfloat16 *q, *k, *v;      // [T][Hq|Hkv][D] packed prompt rows
    const __nv_bfloat16 *wq, *wk;        // [D]
    __nv_bfloat16 *qp;                   // [T][Hq][D] normed + rotated queries
    __nv_bfloat16 *kc, *vc;              // layer base of the cache
    int32_t *lens;                       // layer base of the device lengths
    const float2 *rope;                  // [cap][D/2] (cos, sin)
    uint32_t *err;
    int64_t seq_stride, head_stride;     // cache strides in elements
    int T, Hq, Hkv, cap, nseq;
    int seq_slot0;                       // cache slot of the first sequence of this launch
    int signal_early;                    // 1: let the next kernel (prefill attention) start at once
    float eps;
    int cu[kMaxSeqPerLaunch + 1];        // row offsets of the sequences (relative to q/k/v)
    int start[kMaxSeqPerLaunch];         // position of each sequence's first new token
};

// ---------------------------------------------------------------- K2
constexpr int kK2BlockM = 128;    // query rows per tile
constexpr int kK2BlockN = 128;    // keys per tile

struct alignas(64) K2Params {
    CUtensorMap tm_q;                         // q' [T][Hq][D] as (D, Hq, T)
    CUtensorMap tm_k[kMaxSeqPerLaunch];       // per sequence: (D, start_b + L_b, Hkv) over the cache, 64-row boxes
    CUtensorMap tm_v[kMaxSeqPerLaunch];       // the same with 128-row boxes
    __nv_bfloat16 *out;                       // [T][Hq][D]
    uint32_t *err;
    int nseq, Hq, Hkv, G, npairs;             // npairs: items per kv head and query block
    int hpi;                                  // query heads per item (1, 2, or 4 for a CTA pair; set at launch)
    int len[kMaxSeqPerLaunch];                // new tokens of each sequence
    int start[kMaxSeqPerLaunch];              // position of each sequence's first new token
    int cu[kMaxSeqPerLaunch];                 // first row of each sequence in q'/out
    int max_qblocks;
    int window;                               // attention window in keys (0: all earlier keys)
    float scale_log2;                         // log2(e) / sqrt(D)
    int fault;                                // test hook: withhold a copy in CTA 0 (FaultPlan)
    int nitems;                               // work items (query block x head tile(s))
    uint64_t wait_ns;                         // limit of every bounded wait
};
static_assert(sizeof(K2Params) <= 4096, "K2Params travels in the 4 KB of kernel parameters");

// ---------------------------------------------------------------- K3
constexpr int kK3ConsumerWarps = 5;
constexpr int kK3Chunk = 32;        // keys per pipeline chunk
constexpr int kK3MaxSplits = 16;   // splits of one (sequence, kv head) = CTAs of one cluster
constexpr int kK3MaxSeqPerLaunch = 64;  // positions carried in one launch's parameters
// New tokens per sequence of one launch of the decode kernel family (1 for a
// decode step, up to this many for a short chunk such as a verify step).
constexpr int kK3MaxTokens = 8;
// guard value meaning "every cache row may still be written: load all after the wait"
constexpr int kK3GuardAll = 1 << 30;

struct alignas(64) K3Params {
    // (D, capacity, max_batch * Hkv) over this layer's K / V, in the launch
    // parameters (no descriptor fetch from global memory before the first copy)
    CUtensorMap tmk, tmv;
    const __nv_bfloat16 *q, *k, *v;  // [batch][Hq][D], [batch][Hkv][D] (whole call)
    const __nv_bfloat16 *wq, *wk;
    __nv_bfloat16 *kc, *vc;          // layer base
    int32_t *lens;                   // layer base [max_batch]: set to pos + 1 (null: not kept)
    const float2 *rope;              // [cap][D/2]
    __nv_bfloat16 *out;              // [batch][Hq][D]
    uint32_t *err;
    int64_t seq_stride, head_stride;
    int B, Hq, Hkv, G, HG, cap, S;
    float eps, scale_log2;
    int b0;                          // first sequence of this launch (blockIdx.z = b - b0)
    int window;                      // attention window in keys (0: the whole cache)
    int dev_pos;                     // 0: positions from pos[]; 1: the device lengths, read
                                     // after the launch wait; 2: the device lengths, read at
                                     // once (no launch still running writes this layer)
    int guard;                       // rows just below each sequence's first new slot that
                                     // a launch still running may write (loaded after the wait)
    uint32_t *seq_cnt;               // [max_batch] groups done per sequence (dev_pos only)
    int fault;                       // test hook: withhold a copy in CTA (0,0,0) (FaultPlan)
    uint64_t wait_ns;                // limit of every bounded wait
    int pos[kK3MaxSeqPerLaunch];     // slot of each launched sequence's (first) new token
};

// Per-sequence data of a multi-token launch of the decode kernel (a short
// chunk, e.g. the tokens of a verify step): launched sequence z is cache slot
// seq[z] and holds ntok[z] (1..kK3MaxTokens) new tokens whose rows in q, k,
// v and out start at row0[z]; they take slots pos[z] .. pos[z] + ntok[z] - 1.
struct K3Multi {
    int seq[kK3MaxSeqPerLaunch];
    int ntok[kK3MaxSeqPerLaunch];
    int row0[kK3MaxSeqPerLaunch];
};

}  // namespace qa

#include <cuda_runtime.h>

namespace qa {
// Tensor map of the decode kernel over one layer's K or V: (D, capacity,
// max_batch * Hkv), 64 x 32 x 1 boxes, 128-byte swizzle.  Host-only encode.
bool encode_decode_map(CUtensorMap *m, void *base, int D, int capacity, int rows_z);
// Host launchers, one per kernel file.
cudaError_t launch_k1(const K1Params &p, int D, cudaStream_t stream);
cudaError_t launch_k2(const K2Params &p, int D, int nitems, cudaStream_t stream);
cudaError_t launch_k3(const K3Params &p, int D, int HPC, cudaStream_t stream);
// The multi-token form: p.HG = G / HPC groups of HPC heads, 8 / HPC tokens.
cudaError_t launch_k3_multi(const K3Params &p, const K3Multi &m, int D, int HPC,
                            cudaStream_t stream);
// Number of clusters of S decode CTAs (multi: of the multi-token form) that can
// be resident at once on the current device (cached per device, head_dim,
// form, heads per CTA and S); 0 on error.
int k3_cluster_capacity(int D, int HPC, int S, bool multi);
// Largest split count (<= kK3MaxSplits, <= chunks) such that the clusters of
// `overlap` launches of `groups` clusters each fit on the device at once.
int k3_choose_splits(int D, int HPC, int groups, int pos_max, bool multi, int overlap);
// Upper bound on the CTAs of the decode kernel family resident at once on the
// current device (SMs x the largest per-SM occupancy of any of its kernels).
int k3_max_resident_ctas();
}  // namespace qa
