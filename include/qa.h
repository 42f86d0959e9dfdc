/*
 * qa.h -- C ABI of the GB300 (sm_103a) attention hot path of a greedy
 * Qwen3-style decoder: per-head QK-RMSNorm + rotary embedding + KV-cache
 * append, causal grouped-query prefill attention (whole prompts or chunks
 * appended to what a layer holds; chunks of up to 8 tokens per sequence, such
 * as multi-token verify queries, run in the decode kernel's multi-token form)
 * and decode attention against a preallocated bf16 KV cache, with an optional
 * per-layer attention window.
 *
 * The arguments follow the pages' statement of the problem: a batch of
 * prompts with their lengths, one new token per sequence per decode step,
 * and a cache reset for every generate call (dryft-flash-infer agent guide,
 * sections "What is measured" and "Where the wins are"; the htn.dryft.ai
 * docs, "What to submit", for the Engine.generate contract of one token per
 * sequence per step, sequences kept in arrival order).  Following the
 * pegainfer PR #862 review ("add SM120 FlashInfer GDN prefill candidate",
 * summary and integration-boundary comments), the kernels sit behind a narrow
 * C ABI and an unsupported geometry or invalid argument fails validation with
 * a status code; there is no fallback path of any kind.
 *
 * Conventions for every entry point:
 *  - Tensors are bf16, contiguous, row-major, device pointers, 16-byte
 *    aligned.  The caller owns q, k, v, the norm weights and out; the library
 *    owns the cache, its lengths and its scratch until qa_cache_free.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  All device work is enqueued on it asynchronously; the call
 *    returns once it is enqueued.
 *  - Host-side validation runs before any launch; a call that returns an
 *    error status has enqueued nothing and changed no state.
 *  - Not thread-safe per cache: calls on one cache must come from one thread
 *    (or be serialised by the caller).
 */
#ifndef QA_H_
#define QA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QA_ABI_VERSION 4

typedef enum {
    QA_OK = 0,
    QA_ERR_INVALID_ARG = 1,        /* null pointer, out-of-range layer/batch/length */
    QA_ERR_UNSUPPORTED_SHAPE = 2,  /* head_dim not in {64,128}, Hq % Hkv != 0, group > 8 ... */
    QA_ERR_ALIGNMENT = 3,          /* a tensor pointer is not 16-byte aligned */
    QA_ERR_CAPACITY = 4,           /* a sequence would exceed the cache capacity (no eviction) */
    QA_ERR_STATE = 5,              /* reserved (no current entry point returns it) */
    QA_ERR_CUDA = 6,               /* a CUDA runtime call failed (no device, launch error ...) */
    QA_ERR_DEVICE_TIMEOUT = 7,     /* a kernel gave up a bounded wait (reported by qa_get_device_error) */
    QA_ERR_DEVICE_BOUNDS = 8       /* a kernel saw a position outside the cache (qa_get_device_error) */
} qa_status;

/* Kernels counted by qa_stats (successful launches since qa_cache_alloc). */
enum {
    QA_KERNEL_NORM_ROPE_APPEND = 0, /* K1: fused QK-RMSNorm + RoPE + cache append (prefill rows) */
    QA_KERNEL_PREFILL_ATTN = 1,     /* K2: causal GQA flash attention, TMA + tcgen05 */
    QA_KERNEL_DECODE_ATTN = 2,      /* K3: fused norm/RoPE/append + split-KV decode + LSE merge
                                       (decode steps and short-chunk prefills) */
    QA_KERNEL_RESET = 3,            /* cache-length reset */
    QA_NUM_KERNELS = 4
};

/* Geometry of one cache: num_layers independent layer caches, each holding
 * max_batch sequences of up to `capacity` positions for n_kv_heads heads of
 * head_dim.  Supported: head_dim in {64, 128}; n_q_heads % n_kv_heads == 0
 * with group size n_q_heads / n_kv_heads in {1, 2, 4, 8}; capacity >= 1;
 * rope_theta > 0; rms_eps >= 0. */
typedef struct {
    int num_layers;
    int max_batch;
    int n_q_heads;
    int n_kv_heads;
    int head_dim;
    int capacity;
    float rope_theta;   /* rotary base; angle of pair i at position p is p * theta^(-2i/head_dim) */
    float rms_eps;      /* RMSNorm epsilon, added to the mean of squares */
} qa_config;

typedef struct qa_cache qa_cache; /* opaque */

/* Allocate a cache on the current CUDA device: K and V as bf16
 * [num_layers][max_batch][n_kv_heads][capacity][head_dim] (zero-filled),
 * int32 lengths [num_layers][max_batch] (all zero), an fp32 rotary table
 * [capacity][head_dim/2] of (cos, sin) built on the host in fp64,
 * per-sequence counters and an error word; the decode kernel's TMA tensor
 * maps (two per layer) are kept on the host.  Synchronous.
 * Errors: INVALID_ARG (cfg or out null, non-positive sizes),
 * UNSUPPORTED_SHAPE, CUDA (allocation failed; nothing is leaked). */
qa_status qa_cache_alloc(const qa_config *cfg, qa_cache **out);

/* Free everything qa_cache_alloc allocated.  Synchronises the device first.
 * NULL is accepted and ignored. */
qa_status qa_cache_free(qa_cache *cache);

/* Start a new generate call: every layer's lengths become 0 (device copy on
 * `stream`, host mirror immediately).  K/V memory is not cleared; no kernel
 * ever reads a slot at or beyond its sequence's length. */
qa_status qa_cache_reset(qa_cache *cache, void *stream);

/* Prefill one layer for `batch` prompts (sequence slots 0..batch-1), or the
 * next chunk of them: the L_b = prompt_lens[b] new tokens of sequence b take
 * positions P_b .. P_b + L_b - 1 after the P_b tokens the layer already holds
 * (P_b = 0 after a reset).
 * prompt_lens: HOST array [batch], each >= 0 with P_b + L_b <= capacity.
 * T = sum of L_b.  q: [T][Hq][D], k, v: [T][Hkv][D], packed in sequence order
 * (sequence b's tokens follow sequence b-1's).  q_norm_w, k_norm_w: [D].
 * out: [T][Hq][D]; it also serves as the staging buffer for the normed,
 * rotated queries, so it must not alias q, k or v.
 * Result: k' = RoPE(RMSNorm(k)) and v go to cache slots P_b..P_b+L_b-1, the
 * layer's lengths become P_b + L_b, and for the new token at position i
 * out[t][h] = sum_{j<=i} softmax_j(q'_t,h . K_j / sqrt(D)) V_j over sequence
 * b's cached keys 0..i, q' = RoPE(RMSNorm(q)), kv head h / (Hq/Hkv).
 * Work: when some L_b exceeds 8, K1 writes q' into out and k', v into the
 * cache, then K2 (one launch per 8 sequences) computes the attention.  K2
 * starts its set-up while K1 ends (programmatic dependent launch) and reads
 * or writes global memory only once the kernel before it has finished, so
 * the call is ordered after earlier work on the stream as a plain launch
 * would be.  When
 * every L_b is at most 8 (a verify step of speculative decoding, a short
 * append), the decode kernel's multi-token form does all of it in one launch
 * per 64 sequences that have new tokens (each streams its cache once for all
 * of its new tokens; counted as QA_KERNEL_DECODE_ATTN).  That form overlaps
 * the previous kernel on the stream like qa_decode_step, with the same
 * condition on q, k and v.
 * Errors: INVALID_ARG, ALIGNMENT, CAPACITY (P_b + L_b above capacity). */
qa_status qa_prefill(qa_cache *cache, int layer, int batch, const int32_t *prompt_lens,
                     const void *q, const void *k, const void *v,
                     const void *q_norm_w, const void *k_norm_w, void *out, void *stream);

/* One decode step of one layer: one new token for each of sequences
 * 0..batch-1, at position pos_b = current length of sequence b.
 * q: [batch][Hq][D], k, v: [batch][Hkv][D], weights [D], out: [batch][Hq][D].
 * One fused launch: RMSNorm + RoPE of q and k at pos_b, append of k' and v to
 * slot pos_b, attention of every q head over slots 0..pos_b (the new token
 * attends to itself) split over the key range (the splits of one sequence and
 * kv head form one thread-block cluster), log-sum-exp merge of the splits in
 * distributed shared memory, length += 1 (host copy and device lengths).
 * Positions come from the cache's host copy of the lengths and travel in the
 * launch parameters (one launch per 64 sequences).  Launches may overlap the
 * previous kernel on the stream (programmatic dependent launch): the step
 * reads q, k, v and the weights before that kernel has finished, so they must
 * not be written by the immediately preceding decode step or short chunk (its
 * out buffer in particular must not be this step's q, k or v).  A launch
 * lets the next one start at once, and each of its thread blocks waits for
 * the previous kernel before it exits; the library tracks, per stream, the
 * launches that can still be running when a new one starts (bounded by the
 * thread blocks the device holds at once) and makes the new launch read the
 * cache rows they append to its layer only after its wait.  Kernels of other
 * code enqueued between these calls on the same stream must not let their
 * successors start before they themselves have waited for their predecessor
 * (the usual use of programmatic dependent launch).
 * Errors: INVALID_ARG, ALIGNMENT, CAPACITY (a sequence already holds
 * `capacity` tokens; nothing is evicted or wrapped), CUDA (a launch failed;
 * with more than 64 sequences the launches before it were enqueued and their
 * sequences have advanced, on the device and in the host copy). */
qa_status qa_decode_step(qa_cache *cache, int layer, int batch,
                         const void *q, const void *k, const void *v,
                         const void *q_norm_w, const void *k_norm_w, void *out, void *stream);

/* The same decode step with positions read from the DEVICE lengths, for
 * CUDA-graph capture: a captured step advances the lengths on the device at
 * every replay, so one graph serves every position.  (No counterpart in the
 * pages; it serves the NEXT item "CUDA-graph-captured multi-layer decode step".)
 * Arguments, layouts and ownership as qa_decode_step.  Differences:
 *  - the kernel reads lens[b] from the device: at once when no launch that may
 *    still be running writes this layer (the library's per-stream launch
 *    record says so; e.g. each layer of a captured multi-layer step), and
 *    then it overlaps the previous launch like qa_decode_step; otherwise after
 *    the previous kernel on the stream has finished.  The last kv-head group
 *    of each sequence sets lens[b] + 1 (a per-sequence counter, reset by
 *    qa_cache_reset);
 *  - the host copy of the lengths is not advanced (call qa_cache_sync_lengths
 *    before any call that uses it: qa_prefill, qa_decode_step, the split plan);
 *  - a sequence already at capacity is detected on the device: the step does
 *    nothing for that sequence and qa_get_device_error returns
 *    QA_ERR_DEVICE_BOUNDS;
 *  - the split count is planned for a full cache (capacity) under the cache's
 *    overlap setting (qa_cache_set_decode_overlap), so a captured step and the
 *    same step run eagerly give bit-identical results (any count is correct;
 *    it only sets the speed).
 * Capture requires that the first call on this device for this geometry ran
 * outside capture (it configures the kernel and caches the occupancy query).
 * Errors: INVALID_ARG, ALIGNMENT (host side); DEVICE_BOUNDS (device side). */
qa_status qa_decode_step_device_lengths(qa_cache *cache, int layer, int batch,
                                        const void *q, const void *k, const void *v,
                                        const void *q_norm_w, const void *k_norm_w, void *out,
                                        void *stream);

/* Sliding-window attention for one layer: from now on a token at position i
 * attends to keys max(0, i + 1 - window) .. i in qa_prefill and the decode
 * steps (the new token always included); window = 0 restores attention over
 * all earlier keys (the default).  The cache keeps every key (nothing is
 * evicted); the window only limits what is read.  (No counterpart in the
 * pages' kernels; it serves the NEXT item "sliding-window mask variant".)
 * Host-side only, takes effect for launches after the call.
 * Errors: INVALID_ARG (no such layer, window < 0). */
qa_status qa_cache_set_window(qa_cache *cache, int layer, int window);

/* How many consecutive decode-kernel launches (decode steps, short chunks)
 * the split plan lets run on the device at once.  A launch's split count S
 * is the largest (<= 16) for which `launches` launches' thread-block
 * clusters fit together, so that each launch streams its cache while the
 * next ones start (programmatic dependent launch).
 * Until this is called, each host-position launch chooses from the library's
 * record of the launches on its stream: 1 when nothing may still run beside
 * it (right after a prefill, a reset or a synchronisation through this
 * library), 2 when launches on its own layer may (a single-layer loop), and
 * up to 6 when only other layers' launches may (a loop over attention
 * layers), fewer while 6 would leave a launch a single split (on GB300 this
 * gave the best rate per step at batch 1 and 4 for caches of 512 to 16384
 * keys).  Kernels of other code are not in that record: a caller whose
 * decode launches are separated by other kernels (a model's projections
 * between the attention layers) gets the most splits per launch with 1.
 * Device-length steps always plan for that last case (or the number set
 * here), so a captured step and the same step run eagerly agree bit for bit.
 * Any value gives the same result up to the summation order of the split
 * merge.
 * Host-side only, takes effect for launches after the call.
 * Errors: INVALID_ARG (launches outside 1..8). */
qa_status qa_cache_set_decode_overlap(qa_cache *cache, int launches);

/* Copy one layer's device lengths into the host copy (synchronises `stream`),
 * after decode steps that advanced them on the device. */
qa_status qa_cache_sync_lengths(qa_cache *cache, int layer, void *stream);

/* ---- test and benchmark hooks ------------------------------------------ */

/* Device pointers of one layer's K, V ([max_batch][Hkv][capacity][D] bf16)
 * and lengths ([max_batch] int32), and the element strides of K/V for
 * (sequence, head, position, dim).  Any output pointer may be NULL. */
qa_status qa_cache_view(qa_cache *cache, int layer, void **k, void **v, int32_t **lens,
                        int64_t strides[4]);

/* Overwrite one layer's lengths (HOST array [max_batch], each in
 * [0, capacity]); synchronous with respect to `stream`.  Used to decode
 * against a cache filled through qa_cache_view. */
qa_status qa_cache_set_lengths(qa_cache *cache, int layer, const int32_t *lens_host,
                               void *stream);

/* Copy the host mirror of one layer's lengths into lens_host[max_batch]. */
qa_status qa_cache_lengths(qa_cache *cache, int layer, int32_t *lens_host);

/* Run only K1 of a prefill: like qa_prefill, but the normed, rotated queries
 * go to qprime_out [T][Hq][D] and no attention is computed. */
qa_status qa_prefill_transform(qa_cache *cache, int layer, int batch, const int32_t *prompt_lens,
                               const void *q, const void *k, const void *v,
                               const void *q_norm_w, const void *k_norm_w, void *qprime_out,
                               void *stream);

/* Run only the attention of a prefill (K2): for sequence b, the last
 * prompt_lens[b] positions the layer holds (appended earlier, e.g. by
 * qa_prefill_transform) attend causally to keys 0..own position (and the
 * layer's window), exactly as in qa_prefill.  qprime: [T][Hq][D] normed,
 * rotated queries of those tokens (qa_prefill_transform's output); out:
 * [T][Hq][D]; out may be qprime (in place, as qa_prefill does).  Always the
 * prefill kernel, whatever the lengths.  Splitting qa_prefill this way lets
 * each kernel be timed on its own.  The lengths are not changed.
 * Errors: INVALID_ARG (a prompt_lens[b] above what sequence b holds),
 * ALIGNMENT. */
qa_status qa_prefill_attend(qa_cache *cache, int layer, int batch, const int32_t *prompt_lens,
                            const void *qprime, void *out, void *stream);

/* Synchronise the device, read and clear the error word the kernels set when
 * a bounded wait expired or a position fell outside the cache.  Returns
 * QA_OK, QA_ERR_DEVICE_TIMEOUT or QA_ERR_DEVICE_BOUNDS; *detail (may be NULL)
 * receives the raw word: bits 0-7 kind, 8-15 kernel, 16-31 site. */
qa_status qa_get_device_error(qa_cache *cache, uint32_t *detail);

/* Failure-detection test hook.  Arms the next launch of `kernel`
 * (QA_KERNEL_PREFILL_ATTN, or QA_KERNEL_DECODE_ATTN: decode steps, short
 * chunks and qa_decode_step_noalloc), process-wide: in that launch one tile
 * copy is withheld (prefill: a V tile of the first thread block, or both
 * halves of it in the first CTA pair of the pair form; decode: the first cache
 * chunk of each block of the first sequence's first kv-head group that streams
 * any), so a wait for it can never succeed, and every bounded
 * wait of the launch gives up after wait_us
 * microseconds (1 .. 2000000) instead of 2 s.  The waiting thread records
 * QA_ERR_DEVICE_TIMEOUT (kernel and site in the detail word) in the error
 * word that qa_get_device_error / qa_noalloc_get_device_error read, the block
 * waits (bounded) for its own copies in flight and for what its cluster peers
 * send it, frees its tensor memory and exits; that launch's outputs and the
 * cache slots it appends are undefined, everything else stays usable.
 * kernel = -1 disarms.  Nothing faults or hangs: every wait is bounded.
 * Errors: INVALID_ARG (another kernel index, wait_us out of range). */
qa_status qa_debug_arm_wait_timeout(int kernel, uint32_t wait_us);

/* Successful-launch counters per kernel (QA_KERNEL_*), proving which native
 * kernels ran (the launch-counter check of the pegainfer PR #862 review). */
qa_status qa_stats(qa_cache *cache, uint64_t launches[QA_NUM_KERNELS]);

/* Bytes of device memory the cache owns: K+V, and scratch (device lengths,
 * rotary table, error word). */
qa_status qa_memory_info(qa_cache *cache, uint64_t *kv_bytes, uint64_t *scratch_bytes);

/* Number of key-range splits qa_decode_step uses for the current lengths of
 * `layer` and `batch` sequences when it runs beside other layers' launches
 * (up to 6 launches unless set; see qa_cache_set_decode_overlap;
 * a pure host computation; a step launches one kernel per 64 sequences, and
 * this is the first one's count). */
int qa_decode_splits(qa_cache *cache, int layer, int batch);

/* ---- allocation-free decode step ----------------------------------------
 * The pages have no counterpart of this entry point.  It is for callers that
 * may not allocate device memory at all: engines that hand out every byte of
 * the GPU from their own arena and forbid any other allocation, and plug-ins
 * embedded in a host framework that owns the device allocator.  Such a caller
 * owns the cache memory and the lengths itself and passes them in.
 *
 * One decode step of one layer, computed by the same kernel body as
 * qa_decode_step: for each of sequences 0..batch-1 the new token's q and k are
 * RMS-normed and rotated at position positions[b], k' and v are written to
 * cache slot positions[b], and every query head attends over slots
 * 0..positions[b] (inclusive).
 *   cfg         geometry (num_layers is ignored; one layer is passed).
 *   positions   HOST int32 [batch]: current length of each sequence, which is
 *               the slot of its new token; each must be < capacity.  The
 *               caller advances its own lengths after the call.  The
 *               positions and their rotary values are copied into the
 *               launch's parameters at this call.
 *   k_cache, v_cache  DEVICE bf16 [max_batch][n_kv_heads][capacity][head_dim]
 *               of this layer, caller-owned, read and appended to.
 *   q, k, v, q_norm_w, k_norm_w, out: as in qa_decode_step.
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 * The kernel's only global scratch is its error word (the key-range splits
 * are merged in distributed shared memory), kept in a fixed 256-byte array in
 * the library's device code that every GPU loading the library holds until
 * the process exits.  The first call on a device looks up that array's
 * address (no allocation).
 * Every call shares the array: calls that may overlap on the GPU (different
 * streams without ordering) race on it.  The error word is zero at load and
 * is cleared only by qa_noalloc_get_device_error, so it keeps the first error
 * of any call since the last read.
 * Limits: batch <= 16 (the per-sequence positions and rotary values travel in
 * the kernel parameters), else QA_ERR_UNSUPPORTED_SHAPE.  Errors:
 * INVALID_ARG, UNSUPPORTED_SHAPE, ALIGNMENT, CAPACITY (a position >=
 * capacity), CUDA. */
qa_status qa_decode_step_noalloc(const qa_config *cfg, int batch, const int32_t *positions,
                                 void *k_cache, void *v_cache, const void *q, const void *k,
                                 const void *v, const void *q_norm_w, const void *k_norm_w,
                                 void *out, void *stream);

/* Read and clear the error word of qa_decode_step_noalloc on the current
 * device, after synchronising `stream` (the stream the steps ran on; calls on
 * other streams must have finished too).  Returns QA_OK,
 * QA_ERR_DEVICE_TIMEOUT or QA_ERR_DEVICE_BOUNDS; *detail (may be NULL)
 * receives the raw word (bits 0-7 kind, 8-15 kernel, 16-31 site).  Allocates
 * nothing: a 4-byte copy into host memory and a 4-byte memset.
 * Errors: CUDA. */
qa_status qa_noalloc_get_device_error(uint32_t *detail, void *stream);

/* Static description of a status code. */
const char *qa_status_str(qa_status status);

/* QA_ABI_VERSION of the loaded library. */
int qa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QA_H_ */
