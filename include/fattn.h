/*
 * fattn -- exact softmax-attention forward on GB300 (sm_103a): C ABI.
 *
 * The operation ("FlashAttention-2 in an attention layer", Triton FA2 kernel
 * and launcher; "FlashAttention V2", sections 2-3; "Lecture 6 --
 * FlashAttention-2", Reading task, for the LSE written by the epilogue):
 *
 *   for every batch b, head h and query row i < S:
 *     s_ij   = scale * sum_d Q[b,h,i,d] K[b,h,j,d]   over the allowed keys j
 *              (all j < S; with causal != 0 only j <= i)
 *     O[b,h,i,:] = sum_j softmax_j(s_i.) V[b,h,j,:]
 *     LSE[b,h,i] = max_j s_ij + ln(sum_j exp(s_ij - max_j s_ij))
 *
 * computed tile by tile with an online softmax, so the S x S score matrix
 * never reaches device memory.  Self-attention only: Q, K and V share S.
 *
 * Layout.  q, k, v, o: contiguous [B, H, S, D] row-major 16-bit tensors (D
 * innermost), all of the same dtype.  lse: contiguous [B, H, S] fp32.
 *
 * Ownership.  The caller owns and allocates every buffer (device memory).
 * The library allocates no user-visible memory; it keeps a small per-device
 * status block, two rings of 256 work counters (4 KB) and per-kernel launch
 * attributes for the life of the process.  Outputs may not overlap inputs or
 * each other.
 *
 * Work counters.  A causal fattn_fwd launch at D = 256, and a causal
 * fattn_fwd_fp8 launch or a causal fattn_fwd launch at D = 128 whose K and V
 * (all heads) exceed 32 MiB and split into more than one head group (each
 * group holding at least 1.5 work units per SM), hands its work units out
 * at run time from one
 * counter pair, taken round robin from a ring of 256 per device; the
 * launch's last CTA returns the pair to zero.  Up to 256 such launches may
 * run at once on one device (more would share a pair).  A launch enqueued into a stream capture takes its pair from
 * the second ring and keeps it for every replay of the graph; replays of one
 * graph never overlap, and ordinary launches never use that ring.
 *
 * Asynchrony.  fattn_fwd enqueues the work on ``stream`` and returns; results
 * are visible after the stream is synchronised.
 *
 * Threads.  Every entry point may be called from any host thread; calls on
 * different streams are independent (the no-alloc cache entry excepted, see
 * there).  A call works on the thread's current device; on a thread with no
 * current context it binds that device's primary context to the thread.
 * The device status block is shared by all calls on a device, so a status
 * read by fattn_last_error may come from another thread's call.
 *
 * Errors.  Every entry point returns FATTN_OK (0) or a negative status; none
 * aborts, throws or falls back to another implementation.  Argument errors are
 * detected on the host before anything is enqueued.  An error inside a
 * running kernel (a pipeline wait that exceeded its time limit) is recorded in
 * the device status block; fattn_last_error reads it.
 */
#ifndef FATTN_H_
#define FATTN_H_

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FATTN_API __attribute__((visibility("default")))
#else
#define FATTN_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *fattn_stream_t;

enum fattn_status {
  FATTN_OK = 0,
  FATTN_ERR_INVALID_ARG = -1,      /* null pointer, B/H/S < 1, bad scale,
                                      overlapping buffers, non-device memory
                                      or a buffer smaller than its tensor */
  FATTN_ERR_UNSUPPORTED = -2,      /* D not in {64, 128, 256} (the cache
                                      entry points: {64, 128}), unknown dtype, no
                                      CUDA device, device is not sm_103, or
                                      (cache attention) Sq > 16 */
  FATTN_ERR_MISALIGNED = -3,       /* q/k/v/o not 16-byte aligned, lse not
                                      4-byte aligned */
  FATTN_ERR_TOO_LARGE = -4,        /* B*H*S rows exceed INT32_MAX */
  FATTN_ERR_LAUNCH = -5,           /* the kernel launch failed, or (from
                                      fattn_last_error) the kernel found its
                                      shared memory base misaligned */
  FATTN_ERR_PIPELINE_TIMEOUT = -6, /* a device-side wait exceeded its limit */
  FATTN_ERR_CUDA = -7              /* another CUDA runtime/driver error */
};

enum fattn_dtype { FATTN_FP16 = 0, FATTN_BF16 = 1 };

/*
 * Attention forward: writes o ([B,H,S,D], dtype) and lse ([B,H,S], fp32).
 *   q, k, v  device pointers to the inputs, 16-byte aligned
 *   o        device pointer to the output, 16-byte aligned
 *   lse      device pointer to the fp32 log-sum-exp output, 4-byte aligned
 *   B, H, S  batch, heads, sequence length (each >= 1)
 *   D        head dimension: 64, 128 or 256 (256 runs on pairs of SMs)
 *   causal   0: every key; non-zero: key index <= query index
 *   scale    score multiplier, finite and > 0 (usually 1/sqrt(D))
 *   dtype    FATTN_FP16 or FATTN_BF16 (inputs and output)
 *   stream   CUDA stream to enqueue on
 * Returns FATTN_OK once the kernel is enqueued, else a negative status.
 */
FATTN_API int fattn_fwd(const void *q, const void *k, const void *v, void *o,
                        float *lse, int B, int H, int S, int D, int causal,
                        float scale, int dtype, fattn_stream_t stream);

/*
 * Attention forward with 8-bit inputs ("FlashAttention V2", section 7: FP8
 * attention on the FP8 tensor cores).  The same operation as fattn_fwd on the
 * real values Q = q_scale * Q8, K = k_scale * K8, V = v_scale * V8:
 *   O = softmax(scale * Q K^T [+ causal]) V,  LSE = natural-log LSE of the
 *   scaled scores.
 * Scores and P V run on kind::f8f6f4 tensor-core MMAs; P is rounded to E4M3
 * before the P V product and O is normalised by the sum of those rounded
 * weights (a convex combination of V rows), so O carries the E4M3 rounding
 * of the attention weights (relative 2^-4, absolute 2^-10 below the E4M3
 * normal range, weights taken relative to the row maximum); the LSE uses the
 * fp32 sum of the unrounded weights and does not.
 *
 *   q, k, v    device [B, H, S, D] E4M3 codes (OCP "fn" format: bias 7, three
 *              mantissa bits, largest 448), one byte each, 16-byte aligned
 *   o          device [B, H, S, D] output of out_dtype, 16-byte aligned
 *   lse        device [B, H, S] fp32, 4-byte aligned
 *   D          128
 *   scale      score multiplier on the real values, finite and > 0
 *   q_scale, k_scale, v_scale   per-tensor dequantisation scales, finite > 0
 *   out_dtype  FATTN_FP16 or FATTN_BF16
 * Other arguments, layout, ownership and errors as fattn_fwd.
 */
FATTN_API int fattn_fwd_fp8(const void *q, const void *k, const void *v, void *o,
                            float *lse, int B, int H, int S, int D, int causal,
                            float scale, float q_scale, float k_scale,
                            float v_scale, int out_dtype, fattn_stream_t stream);

/*
 * Synchronises ``stream``, then reads and clears the current device's status
 * block.  Returns FATTN_OK, FATTN_ERR_PIPELINE_TIMEOUT (a kernel gave up on a
 * wait and unwound; its outputs are incomplete), FATTN_ERR_LAUNCH (a kernel
 * did not run because its shared memory base was not 1024-byte aligned),
 * FATTN_ERR_INVALID_ARG (fattn_fwd_kvcache met a cached length outside
 * [0, Sk]) or FATTN_ERR_CUDA when the synchronisation itself reported an
 * error.  ``detail`` (may be NULL)
 * receives where the kernel error was raised: detail[0] = role << 8 |
 * barrier, detail[1] = block index.
 */
FATTN_API int fattn_last_error(fattn_stream_t stream, int *detail);

/*
 * Checks the device-side bounded wait the kernels use: one warp waits on a
 * shared-memory barrier that nothing completes, with a limit of timeout_us
 * microseconds (1 .. 1000000); it gives up, records
 * FATTN_ERR_PIPELINE_TIMEOUT in the device status block (detail[0] = 7 << 8)
 * and exits, leaving the context usable.  Enqueued on ``stream``; read the
 * outcome with fattn_last_error.  Returns FATTN_OK once enqueued,
 * FATTN_ERR_INVALID_ARG for a limit out of range, or the device errors of
 * fattn_fwd.
 */
FATTN_API int fattn_check_wait_timeout(int timeout_us, fattn_stream_t stream);

/* A static, human-readable string for a status code. */
FATTN_API const char *fattn_error_string(int status);

/*
 * The launch fattn_fwd would make for these sizes, without launching.
 * Fills (each pointer may be NULL): grid (CTAs), block (threads), dynamic
 * shared memory bytes, work units (query-tile groups over all heads), query
 * tiles of 128 rows per unit, and K/V pipeline stages.  For D = 256 a unit is
 * served by a cluster of two CTAs (one query tile each) and the grid counts
 * CTAs.  Needs a device only for the grid (it depends on the SM count and,
 * for D = 256, on how many clusters fit); without one *grid is set to the
 * number of CTAs the units would use.  Returns FATTN_OK or the status
 * fattn_fwd would return for the same sizes' host-side checks.
 */
FATTN_API int fattn_plan(int B, int H, int S, int D, int causal, int *grid,
                         int *block, int *smem_bytes, int *units,
                         int *q_tiles_per_unit, int *kv_stages);

/*
 * The order in which a causal launch of these sizes takes its work units on
 * a device with ``sms`` SMs, without a device (the persistent grid of the
 * "Lecture 6" FA2 change 1, parallelism over the sequence, longest units
 * first).  elem_bytes is 2 for fattn_fwd (fp16/bf16) and 1 for fattn_fwd_fp8
 * (D = 128).  Fills (each pointer may be NULL): *group_heads, the heads of
 * one group of the order (B*H when every head is in one group; the groups
 * differ by at most one head), and *run_time, 1 when the units are handed
 * out at run time from a per-launch counter, 0 when each CTA takes the
 * static longest-first snake.  Returns FATTN_OK, FATTN_ERR_INVALID_ARG (sms
 * < 1, elem_bytes not 1 or 2), FATTN_ERR_UNSUPPORTED (E4M3 with D != 128)
 * or the status fattn_plan returns for the same sizes.
 */
FATTN_API int fattn_causal_order(int B, int H, int S, int D, int elem_bytes,
                                 int sms, int *group_heads, int *run_time);

/*
 * Attention of a few new queries against a key/value cache ("FlashAttention
 * V2", section 6: inference with a KV cache, which FlashAttention serves with
 * its decoding variant; the per-row recurrence of section 3).
 *
 * For batch b, head h: the cache holds len_b positions (rows 0 .. len_b-1 of
 * the [B, H, Sk, D] caches; Sk is the capacity, rows at or past len_b are
 * ignored whatever they hold).  The Sq new queries are the last Sq positions
 * of the sequence: query i sits at position len_b - Sq + i and attends to
 * every key j < len_b, or with causal != 0 only to j <= len_b - Sq + i.
 *   O[b,h,i,:] = sum_j softmax_j(scale * q_i . k_j) V[b,h,j,:]
 *   LSE[b,h,i] = m + ln(sum_j exp(s_ij - m))
 * A query with no allowed key (len_b = 0, or causal with len_b < Sq - i)
 * gets O = 0 and LSE = -inf.
 *
 * The keys are split across every warp of the GPU; each slice writes a
 * partial (O, LSE) record to ``workspace`` and a second kernel merges a
 * head's records with weights exp(LSE_s - max LSE).  Both kernels are
 * enqueued on ``stream``.
 *
 *   q          device [B, H, Sq, D] 16-bit, 16-byte aligned
 *   k_cache    device [B, H, Sk, D] 16-bit, 16-byte aligned
 *   v_cache    device [B, H, Sk, D] 16-bit, 16-byte aligned
 *   cache_lens device int32 [B] cached lengths in [0, Sk], 4-byte aligned, or
 *              NULL for every length equal to Sk.  A value outside [0, Sk]
 *              is clamped for memory safety and reported by
 *              fattn_last_error as FATTN_ERR_INVALID_ARG (detail[0] = 6 << 8,
 *              detail[1] = the batch index); the outputs are then undefined.
 *              The lengths must not change while the call runs (the kernels
 *              read them several times); if they do, the kernels stop
 *              without reading outside any buffer, report
 *              FATTN_ERR_INVALID_ARG (detail[0] = 6 << 8 | 1) and leave the
 *              outputs undefined.
 *   o          device [B, H, Sq, D] 16-bit output, 16-byte aligned
 *   lse        device [B, H, Sq] fp32 output, 4-byte aligned
 *   B, H       batch and heads (>= 1)
 *   Sq         new queries per head: 1 .. 16
 *   Sk         cache capacity (>= 1)
 *   D          head dimension: 64 or 128
 *   causal     0: every cached key; non-zero: keys up to each query's position
 *   scale      score multiplier, finite and > 0
 *   dtype      FATTN_FP16 or FATTN_BF16 (q, caches and o)
 *   workspace  device scratch of at least the size fattn_kvcache_plan gives
 *              for these sizes on the current device, 16-byte aligned; owned
 *              by the caller; its contents need no initialisation and are
 *              meaningless afterwards.  Calls in flight at the same time need
 *              separate workspaces.
 *   workspace_bytes  its size in bytes
 * Outputs (o, lse, workspace) may not overlap the inputs or each other.
 * Returns FATTN_OK once both kernels are enqueued, else a negative status
 * (FATTN_ERR_UNSUPPORTED for Sq > 16 or D not in {64, 128};
 * FATTN_ERR_INVALID_ARG also for a workspace that is too small).
 */
FATTN_API int fattn_fwd_kvcache(const void *q, const void *k_cache,
                                const void *v_cache, const int *cache_lens,
                                void *o, float *lse, int B, int H, int Sq,
                                int Sk, int D, int causal, float scale,
                                int dtype, void *workspace,
                                unsigned long long workspace_bytes,
                                fattn_stream_t stream);

/*
 * The launch fattn_fwd_kvcache would make for these sizes on the current
 * device, without launching.  Fills (each pointer may be NULL): the
 * workspace bytes it needs, the split kernel's grid (CTAs), block (threads)
 * and dynamic shared memory, and the total number of split warps.  Needs a
 * device (the split depends on its SM count).  Returns FATTN_OK or the
 * status fattn_fwd_kvcache would return for the same sizes.
 */
FATTN_API int fattn_kvcache_plan(int B, int H, int Sq, int Sk, int D,
                                 unsigned long long *workspace_bytes,
                                 int *grid, int *block, int *smem_bytes,
                                 int *split_warps);

/*
 * fattn_fwd_kvcache without any device allocation, for callers that cannot
 * call cudaMalloc.  The pages have no counterpart to this entry point: it is
 * the same computation as fattn_fwd_kvcache (same kernels, same split, same
 * results), with the split partials kept in a file-scope static device array
 * of FATTN_NOALLOC_SCRATCH_BYTES instead of a caller workspace.
 *
 * Limit.  The scratch holds (split warps + B*H) * Sq * (D + 1) fp32 values
 * (fattn_kvcache_plan's workspace_bytes); a call needing more than
 * FATTN_NOALLOC_SCRATCH_BYTES returns FATTN_ERR_TOO_LARGE before anything is
 * enqueued.  The scratch needs no clearing: every value the merge kernel
 * reads is written by the split kernel of the same call.
 *
 * First call.  The first call on a device (the current device) queries it
 * and takes the scratch's address with cudaGetSymbolAddress (its return code
 * checked; failure gives FATTN_ERR_CUDA); make that first call before any
 * stream capture begins.  No call allocates device or host memory.
 *
 * Concurrency.  Calls on one device share the one scratch array: calls whose
 * kernels overlap in time (other streams, or other host threads) race on it
 * and give undefined results.  Calls in order on one stream are safe.
 *
 * status_words: device pointer to 4 ints that start at zero (the caller clears
 * them), or NULL.  Kernel-side errors of this call (a cached length outside
 * [0, Sk], a pipeline wait past its limit) are recorded there as
 * fattn_last_error would report them: word 0 the status, word 1 where, word 2
 * the block or batch index.  With NULL they go to a private static word that
 * is never read: fattn_last_error does not see errors of this entry point in
 * either case, so a caller that needs them passes status_words.
 *
 * Every other argument, layout and return code as fattn_fwd_kvcache.
 */
#define FATTN_NOALLOC_SCRATCH_BYTES (32ull << 20)

FATTN_API int fattn_fwd_kvcache_noalloc(const void *q, const void *k_cache,
                                        const void *v_cache,
                                        const int *cache_lens, void *o,
                                        float *lse, int B, int H, int Sq,
                                        int Sk, int D, int causal, float scale,
                                        int dtype, int *status_words,
                                        fattn_stream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
FATTN_API int fattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H_ */
