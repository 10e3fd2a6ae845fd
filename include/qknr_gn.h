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
 * rounded once into the activation dtype.  The statistics are fp32: each
 * thread sums x - k and (x - k)^2 around its own first value k, which gives
 * its count, its mean and its sum of squared deviations; these parts are
 * merged around the mean of one of them, in each warp, across a piece's
 * warps and across a group's pieces, so neither an outlier nor a large mean
 * cancels the variance away.  With K the lower median of the group's
 * first 8 values (one of its values, among the bulk unless 4 of those 8
 * are outliers) and m1 = mean - K, the output is formed from x - K, as
 * (x - K) * a + (beta - m1 * a) with a = gamma * rsqrt(var + eps), so a
 * group whose mean is large against its spread keeps its small differences
 * (x - K is exact for nearby values).
 *
 * A group is large and there are few of them, so each is cut into pieces
 * whose statistics go to a caller-provided device workspace.  Two paths:
 *
 *   fused (QKNR_GN_FUSED): one persistent cooperative launch, one CTA per
 *     SM, that reads x once.  Each 12288-element piece is kept in shared
 *     memory from its statistics to its normalise + SiLU pass; CTAs publish
 *     piece statistics through the workspace, tagged with a value unique to
 *     the call (so the workspace needs no clearing), and wait (bounded) for
 *     the other pieces of a group.  A call made while its stream is being
 *     captured into a CUDA graph adds a memset of the records before the
 *     launch, so every replay starts clean.  Needs cooperative launch support and
 *     groups of at most 9 * SMs pieces (16.8 M elements on 152 SMs).
 *   two-pass (QKNR_GN_TWO_PASS): a statistics kernel and a normalise + SiLU
 *     kernel, once for all groups or once per batch of groups; x is read
 *     twice.  No CTA waits for another.
 *   cluster (QKNR_GN_CLUSTER): one thread-block cluster (up to 16 CTAs) per
 *     group of a sample; each CTA holds an equal part of the group in
 *     shared memory, the parts' statistics are merged over distributed
 *     shared memory in one fixed order, and each CTA writes its own part:
 *     x read once, no workspace (qknr_gn_workspace_bytes reports 0), no CTA
 *     waits outside its cluster.  Needs cluster launch support and groups
 *     whose parts fit 200 KB of shared memory at 16 CTAs (about 1.6 M
 *     elements); a CTA's copy wait is bounded like the fused path's.
 *
 * QKNR_GN_AUTO, when piece_elems and l2_batch_bytes are 0 (they tune the
 * two-pass path), takes the cluster path for groups of at most 512 KB
 * (parts of at most 32 KB) when the device can place all the call's
 * clusters at once, else
 * the fused path when this device and shape allow it, else the two-pass
 * path; it also falls back to the two-pass path when the cooperative
 * launch does not fit the SMs the context may use.  The fused and two-pass
 * paths give the same bits when the two-pass pieces are 12288 elements;
 * the cluster path sums in other parts, so its bits differ from theirs
 * within the same tolerance (and equal them when one CTA holds a group).
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

typedef enum {
  QKNR_GN_AUTO = 0,
  QKNR_GN_FUSED = 1,          /* QKNR_ERR_UNSUPPORTED where the fused path cannot run */
  QKNR_GN_TWO_PASS = 2,
  QKNR_GN_CLUSTER = 3         /* QKNR_ERR_UNSUPPORTED where the cluster path cannot run */
} qknr_gn_mode;

/* test only: the fused path publishes no piece statistics, so every wait
   for a group's statistics runs out and the call reports QKNR_ERR_TIMEOUT */
#define QKNR_GN_FLAG_TEST_NO_RECORDS 0x2u

typedef struct qknr_gn_args {
  uint32_t abi_version;       /* QKNR_ABI_VERSION */
  int32_t dtype;              /* QKNR_BF16 or QKNR_FP16 */
  const void *x;              /* device [N, C, H, W], contiguous */
  void *out;                  /* device [N, C, H, W]; NULL or x = in place */
  int32_t n, c, h, w;         /* > 0; H*W a multiple of 8; (C/G)*H*W < 2^31 */
  int32_t groups;             /* G, divides C */
  const float *gamma, *beta;  /* device fp32 [C] */
  float eps;                  /* default 1e-6 */
  void *workspace;            /* device, 16-byte aligned, qknr_gn_workspace_bytes() (NULL when 0) */
  size_t workspace_bytes;
  int32_t piece_elems;        /* elements per piece (multiple of 8); 0 = about 1024 pieces in all, >= 65536 each */
  int64_t l2_batch_bytes;     /* activation bytes per batch of groups; 0 or -1 = one batch */
  int32_t *dev_status;        /* optional device int32: the fused path writes QKNR_ERR_TIMEOUT
                                 here when one of its waits runs out (see qknr.h) */
  int32_t mode;               /* QKNR_GN_AUTO, QKNR_GN_FUSED, QKNR_GN_TWO_PASS or QKNR_GN_CLUSTER */
  uint32_t flags;             /* QKNR_FLAG_TEST_STALL, QKNR_GN_FLAG_TEST_NO_RECORDS (tests only) */
  uint64_t wait_limit_ns;     /* bound of each wait of the fused path; 0 = 2 s */
} qknr_gn_args;

/* Defaults: bf16, eps 1e-6, automatic pieces and batches, all else zero. */
void qknr_gn_args_init(qknr_gn_args *a);

/* Device workspace the call needs for these arguments: 16 bytes per piece
   and one more per group of each sample, plus 16 bytes for the fused path
   (in QKNR_GN_AUTO the larger of the fused and two-pass paths' needs,
   since it may fall back to either); 0 in QKNR_GN_CLUSTER, where workspace
   may be NULL.
   Depends on the arguments only, not on the device. */
qknr_status qknr_gn_workspace_bytes(const qknr_gn_args *args, size_t *bytes);

/* Validate and launch on `stream` (asynchronous). */
qknr_status qknr_gn_silu_forward(const qknr_gn_args *args, qknr_stream_t stream);

/* Validate and describe the launch without launching: for the fused path
   the grid, block, shared memory, ring slots (stages) and piece bytes
   (stage_bytes); for the two-pass path the apply kernel's grid (pieces x
   groups of a batch) and block; for the cluster path the grid, block,
   shared memory and part bytes, with the CTAs per cluster in `kernel`.
   Queries the current device. */
qknr_status qknr_gn_query(const qknr_gn_args *args, qknr_launch_info *info);

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
 * that device current) and caches it for the life of the process; make
 * that first call before any stream capture.  The cached address belongs
 * to the context that was current then: after cudaDeviceReset() (or with
 * another context made current on that device) the library's module is
 * loaded again at an address the cache does not know, so do not use this
 * entry point in a process that resets a device it has already used it
 * on.  Every call on a device shares the one array, and
 * nothing in it needs clearing: the two-pass path reads only what the same
 * call wrote, and the fused path accepts only statistics tagged with its
 * own call's tag; the cluster path does not touch it.  Calls whose kernels
 * overlap on the GPU (different streams, no ordering between them) race on
 * the array, except on the cluster path.
 */
#define QKNR_GN_NOALLOC_SCRATCH_BYTES (1 << 20)
qknr_status qknr_gn_silu_forward_noalloc(const qknr_gn_args *args, qknr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QKNR_GN_H_ */
