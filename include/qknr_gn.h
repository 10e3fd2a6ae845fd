/*
 * qknr_gn.h — C ABI of the group-norm + SiLU kernels in libqknr.so.
 *
 * "fused qknorm rope Flux 2.0" (TensorRT-Model-Connect PR #239, section
 * "Not in this PR — follow-ups") lists group_norm_silu for the VAE.  For
 * an NCHW activation x [N, C, H, W] with G groups (C/G channels each), per
 * sample n and group g, over the (C/G)*H*W elements of that group:
 *
 *     mean, var = mean and biased variance of the group's elements
 *     y[c, h, w] = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c]
 *     out = y * sigmoid(y) = y / (1 + exp(-y))
 *
 * rounded once into the activation dtype.  The statistics are sums around
 * the group's first element K, S1 = sum (x - K), S2 = sum (x - K)^2, taken
 * per piece in fp32 and combined in fp64: mean = K + S1/L, var = S2/L -
 * (S1/L)^2.
 *
 * A group is large and there are few of them, so each is cut into pieces
 * and the call runs two stream-ordered kernels (piece statistics into a
 * caller-provided device workspace, then the normalise + SiLU pass), once
 * for all groups or once per batch of groups.  No kernel waits for another
 * CTA.
 *
 * Ownership and errors follow qknr.h: the caller owns every buffer
 * (activations, gamma, beta and the workspace); the library allocates
 * nothing and never synchronises; argument errors return before any CUDA
 * call.  Two calls that share a workspace must not run concurrently.
 */
#ifndef QKNR_GN_H_
#define QKNR_GN_H_

#include "qknr.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct qknr_gn_args {
  uint32_t abi_version;       /* QKNR_ABI_VERSION */
  int32_t dtype;              /* QKNR_BF16 or QKNR_FP16 */
  const void *x;              /* device [N, C, H, W], contiguous */
  void *out;                  /* device [N, C, H, W]; NULL or x = in place */
  int32_t n, c, h, w;         /* > 0; H*W a multiple of 8; (C/G)*H*W < 2^31 */
  int32_t groups;             /* G, divides C */
  const float *gamma, *beta;  /* device fp32 [C] */
  float eps;                  /* default 1e-6 */
  void *workspace;            /* device, 16-byte aligned, qknr_gn_workspace_bytes() */
  size_t workspace_bytes;
  int32_t piece_elems;        /* elements per piece (multiple of 8); 0 = about 1024 pieces in all, >= 65536 each */
  int64_t l2_batch_bytes;     /* activation bytes per batch of groups; 0 or -1 = one batch */
} qknr_gn_args;

/* Defaults: bf16, eps 1e-6, automatic pieces and batches, all else zero. */
void qknr_gn_args_init(qknr_gn_args *a);

/* Device workspace the call needs for these arguments (16 bytes per piece
   and one more per group of each sample). */
qknr_status qknr_gn_workspace_bytes(const qknr_gn_args *args, size_t *bytes);

/* Validate and launch on `stream` (asynchronous). */
qknr_status qknr_gn_silu_forward(const qknr_gn_args *args, qknr_stream_t stream);

/* sizeof(qknr_gn_args) as compiled into the library. */
size_t qknr_gn_sizeof_args(void);

/*
 * The same operation for callers that cannot allocate device memory — a
 * plugin or runtime with no allocator on its execution path, a fixed
 * device-memory budget, or a workspace size fixed before the shapes were
 * known.  The pages have no counterpart of this entry point.
 *
 * It ignores args->workspace and args->workspace_bytes: the statistics go
 * to a fixed array of QKNR_GN_NOALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library holds until the process exits.
 * A shape whose qknr_gn_workspace_bytes() exceeds that size is rejected
 * with QKNR_ERR_UNSUPPORTED before anything runs (larger pieces need
 * fewer bytes).  It calls no allocator.
 *
 * The first call on a device looks up the array's device address (with
 * that device current) and caches it; make that first call before any
 * stream capture.  Every call on a device shares the one array and every
 * call writes all the scratch it reads, so nothing needs clearing, but
 * calls whose kernels overlap on the GPU (different streams, no ordering
 * between them) race on it.
 */
#define QKNR_GN_NOALLOC_SCRATCH_BYTES (1 << 20)
qknr_status qknr_gn_silu_forward_noalloc(const qknr_gn_args *args, qknr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QKNR_GN_H_ */
