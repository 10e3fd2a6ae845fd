/*
 * qknr_adaln.h — C ABI of the AdaLN scale/shift kernel in libqknr.so.
 *
 * "fused qknorm rope Flux 2.0" (TensorRT-Model-Connect PR #239, section
 * "Not in this PR — follow-ups") names AdaLN's fuse_scale_shift, called 81
 * times per FLUX.2 step, as the next fusion.  Read plainly, it is adaptive
 * layer normalisation: for every token row t of a hidden state x [T, C]
 * belonging to sample b = t / rows_per_batch,
 *
 *     mean = sum_c x[c] / C,   var = sum_c (x[c] - mean)^2 / C
 *     out[c] = (x[c] - mean) * rsqrt(var + eps) * (1 + scale[b, c]) + shift[b, c]
 *
 * rounded once, to nearest even, into the activation dtype.  The kernel
 * takes mean and variance in fp32 from one pass over the row: each thread
 * sums x - k and (x - k)^2 around its own first value k, and the threads'
 * counts, means and sums of squared deviations are merged around the mean
 * of one of them, so neither an outlier channel nor a large mean cancels
 * the variance away.  With K the lower median of x[0..7] (one of the row's
 * values, among the bulk unless 4 of those 8 are outliers) and m1 = mean -
 * K, it normalises as (x - K) * r - m1 * r with r = rsqrt(var + eps), so a
 * row whose mean is large against its spread keeps its small differences
 * (x - K is exact for nearby values).
 *
 * Ownership and errors follow qknr.h: the caller owns every buffer, the
 * library allocates nothing and never synchronises; argument errors return
 * before any CUDA call; a bounded in-kernel wait that runs out writes
 * QKNR_ERR_TIMEOUT to *dev_status.
 */
#ifndef QKNR_ADALN_H_
#define QKNR_ADALN_H_

#include "qknr.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct qknr_adaln_args {
  uint32_t abi_version;       /* QKNR_ABI_VERSION */
  int32_t dtype;              /* activations x and out: QKNR_BF16 or QKNR_FP16 */
  const void *x;              /* device [T, C], row stride x_stride elements */
  void *out;                  /* device [T, C]; NULL or x (same stride) = in place */
  int64_t x_stride, out_stride;   /* elements per row; 0 = C (out: x's) */
  int64_t tokens;             /* T; 0 is a no-op */
  int32_t hidden;             /* C: a multiple of 8, at most 32768 */
  int64_t rows_per_batch;     /* rows sharing one modulation row; 0 = tokens */
  const void *scale, *shift;  /* device [B, C], B = ceil(T / rows_per_batch) */
  int32_t mod_dtype;          /* QKNR_FP32, or the activation dtype */
  int64_t mod_stride;         /* elements between samples' rows; 0 = C */
  float eps;                  /* default 1e-6 */
  int32_t *dev_status;        /* optional device int32 (see qknr.h) */
  /* launch tuning; 0 = automatic */
  int32_t ctas_per_sm, stages, consumer_warps, group_warps;
  uint32_t flags;             /* QKNR_FLAG_* */
  uint64_t wait_limit_ns;     /* 0 = 2 s */
} qknr_adaln_args;

/* Defaults: bf16, fp32-free (mod_dtype = activation dtype), eps 1e-6,
   automatic tuning, everything else zero. */
void qknr_adaln_args_init(qknr_adaln_args *a);

/* Validate and launch on `stream` (asynchronous).  Base addresses, row and
   sample strides must be 16-byte aligned; `out` must not partially overlap
   x, scale or shift.  Launched like qknr_forward (programmatic dependent
   launch unless flags has QKNR_FLAG_NO_OVERLAP); before its wait for the
   previous kernel each CTA only asks L2 to prefetch its first four rows of
   x (QKNR_FLAG_NO_PREFETCH skips that; qknr_launch_info.prefetch_rows
   reports it). */
qknr_status qknr_adaln_forward(const qknr_adaln_args *args, qknr_stream_t stream);

/* Validate and describe the launch without launching. */
qknr_status qknr_adaln_query(const qknr_adaln_args *args, qknr_launch_info *info);

/* sizeof(qknr_adaln_args) as compiled into the library. */
size_t qknr_adaln_sizeof_args(void);

#ifdef __cplusplus
}
#endif

#endif /* QKNR_ADALN_H_ */
