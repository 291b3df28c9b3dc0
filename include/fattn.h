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
 * status block and per-kernel launch attributes for the life of the process.
 * Outputs may not overlap inputs or each other.
 *
 * Asynchrony.  fattn_fwd enqueues the work on ``stream`` and returns; results
 * are visible after the stream is synchronised.
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
  FATTN_ERR_UNSUPPORTED = -2,      /* D not in {64, 128}, unknown dtype, no
                                      CUDA device, or device is not sm_103 */
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
 *   D        head dimension: 64 or 128
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
 * Synchronises ``stream``, then reads and clears the current device's status
 * block.  Returns FATTN_OK, FATTN_ERR_PIPELINE_TIMEOUT (a kernel gave up on a
 * wait and unwound; its outputs are incomplete), FATTN_ERR_LAUNCH (a kernel
 * did not run because its shared memory base was not 1024-byte aligned) or
 * FATTN_ERR_CUDA when the synchronisation itself reported an error.  ``detail`` (may be NULL)
 * receives where the kernel error was raised: detail[0] = role << 8 |
 * barrier, detail[1] = block index.
 */
FATTN_API int fattn_last_error(fattn_stream_t stream, int *detail);

/* A static, human-readable string for a status code. */
FATTN_API const char *fattn_error_string(int status);

/*
 * The launch fattn_fwd would make for these sizes, without launching.
 * Fills (each pointer may be NULL): grid (CTAs), block (threads), dynamic
 * shared memory bytes, work units (query-tile groups over all heads), query
 * tiles of 128 rows per unit, and K/V pipeline stages.  Needs a device only
 * for the grid (it depends on the SM count); without one *grid is set to the
 * number of units.  Returns FATTN_OK or the status fattn_fwd would return
 * for the same sizes' host-side checks.
 */
FATTN_API int fattn_plan(int B, int H, int S, int D, int causal, int *grid,
                         int *block, int *smem_bytes, int *units,
                         int *q_tiles_per_unit, int *kv_stages);

/* Library version: major * 10000 + minor * 100 + patch. */
FATTN_API int fattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H_ */
