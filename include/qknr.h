/*
 * qknr.h — C ABI of the fused DiT QK-RMSNorm + RoPE library (libqknr.so).
 *
 * The operation, per token row t of a Q/K/V activation, follows two pages:
 *
 *  - "fused qknorm rope Flux 2.0" (TensorRT-Model-Connect PR #239, title
 *    section): one fused call replaces each block's per-head RMSNorms and
 *    the RoPEs that follow them; the kernel is templated on the activation
 *    dtype (fp16 and bf16) and can be launched once per tensor.
 *  - "VisualGen Wan: deduplicate shared RoPE SMEM staging" (TensorRT-LLM
 *    PR #18036, Description and Test Coverage): one cos/sin row per token
 *    is staged once and indexed by dimension for every head; the per-head
 *    expanded table must give the same bits; the V slice is unchanged.
 *
 * For each head h of Q (gain gamma_q) and of K (gain gamma_k), with
 * x = the head's D input values widened to fp32:
 *
 *     r    = rsqrt(sum_d x[d]^2 / D + eps)               (fp32)
 *     y[d] = x[d] * r * gamma[d]
 *     o[d] = y[d] * cos[d] + s(d) * y[p(d)] * sin[d]
 *
 * p(d) is d's rotation partner: d xor 1 for interleaved pairing, d +/- D/2
 * for rotate-half.  s(d) is -1 for the first member of a pair (even d;
 * d < D/2) and +1 for the second.  The result is rounded once, to nearest
 * even, into the activation dtype.  V is either left alone or copied
 * bit for bit.  The kernel evaluates o[d] as r * (x[d]*a[d] + x[p]*b[d])
 * with a[d] = gamma[d]*cos[d] and b[d] = s(d)*gamma[p]*sin[d], each
 * product rounded in fp32, so shared and expanded tables of equal values
 * give bitwise-equal outputs.
 *
 * Ownership: the caller owns every buffer.  The library allocates no
 * memory and never synchronises the stream.  Between calls it keeps only
 * what it looks up once and caches: device attributes, a per-kernel
 * "max dynamic shared memory" attribute it sets, and occupancy queries.
 */
#ifndef QKNR_H_
#define QKNR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *qknr_stream_t;

#define QKNR_ABI_VERSION 3

typedef enum {
  QKNR_BF16 = 0, /* activations or cos/sin */
  QKNR_FP16 = 1, /* activations only */
  QKNR_FP32 = 2  /* cos/sin only */
} qknr_dtype;

typedef enum {
  QKNR_ROPE_INTERLEAVED = 0, /* pairs (2i, 2i+1) */
  QKNR_ROPE_ROTATE_HALF = 1  /* pairs (i, i + D/2) */
} qknr_rope_style;

typedef enum {
  /* cos, sin: [cos_rows, D]; token t reads row t % cos_rows for all heads */
  QKNR_COS_SHARED_ROW = 0,
  /* cos, sin: [cos_rows, H, D]; head h of Q and head h of K read [t % cos_rows, h] */
  QKNR_COS_PER_HEAD_EXPANDED = 1
} qknr_cos_layout;

typedef enum {
  QKNR_OK = 0,
  QKNR_ERR_NULL = 1,        /* a required pointer is NULL */
  QKNR_ERR_SHAPE = 2,       /* a size, count or stride is out of range */
  QKNR_ERR_ALIGN = 3,       /* a base address or row stride is not 16-byte aligned */
  QKNR_ERR_UNSUPPORTED = 4, /* valid request the library does not implement */
  QKNR_ERR_CUDA = 5,        /* a CUDA runtime call failed; see qknr_last_error() */
  QKNR_ERR_TIMEOUT = 6,     /* written to *dev_status by a kernel whose wait ran out */
  QKNR_ERR_OVERLAP = 7,     /* an output partially overlaps an input */
  QKNR_ERR_ABI = 8,         /* args->abi_version != QKNR_ABI_VERSION */
  QKNR_ERR_BOUNDS = 9       /* written to *dev_status by a kernel of the checked build
                               (libqknr_checked.so) that found an access outside its
                               buffers; the access was skipped */
} qknr_status;

/* Launch-time flags (qknr_args.flags). */
#define QKNR_FLAG_TEST_STALL 0x1u /* test only: issue no loads, so every wait runs out
                                     and the kernel reports QKNR_ERR_TIMEOUT */
#define QKNR_FLAG_NO_OVERLAP 0x2u /* launch without programmatic dependent launch and
                                     without the early L2 prefetch (see qknr_forward) */
#define QKNR_FLAG_NO_PREFETCH 0x8u /* keep programmatic dependent launch but skip the L2
                                      prefetch before the dependency wait (see
                                      qknr_forward) */
#define QKNR_FLAG_TEST_SHORT_OUT 0x4u /* test only, checked build: the Q output span its
                                         kernel checks against ends one row early, so the
                                         last row's Q stores are refused and reported as
                                         QKNR_ERR_BOUNDS (ignored by the regular build) */

/*
 * Arguments of one call.  Fill with qknr_args_init() and then set fields.
 *
 * Activations are row-major with one row per token; a row holds the heads
 * of that tensor back to back (head h at elements [h*D, (h+1)*D)).
 *  - Packed QKV [T, (Hq+Hk+Hv)*D]: q = base, k = base + Hq*D elements,
 *    v = base + (Hq+Hk)*D elements, all three strides (Hq+Hk+Hv)*D.
 *  - Separate tensors [T, H*D]: stride H*D (or 0, meaning H*D).
 *  - Per-tensor launch (page 2's form): set only one of q / k and give the
 *    other zero heads.
 *
 * Strides are in elements.  Every base address and every stride in bytes
 * must be a multiple of 16 (QKNR_ERR_ALIGN otherwise).
 *
 * q_out / k_out NULL, or equal to q / k with the same stride, means in
 * place.  V is copied only when v_out is non-NULL, differs from v and
 * n_heads_v > 0; otherwise it is not touched.  An output that is not its
 * own input must not overlap any input (QKNR_ERR_OVERLAP).
 */
typedef struct qknr_args {
  uint32_t abi_version;       /* QKNR_ABI_VERSION */
  int32_t dtype;              /* qknr_dtype of q, k, v and outputs: BF16 or FP16 */

  const void *q, *k, *v;      /* device pointers; unused ones may be NULL */
  void *q_out, *k_out, *v_out;
  int64_t q_stride, k_stride, v_stride;             /* elements per row; 0 = H*D */
  int64_t q_out_stride, k_out_stride, v_out_stride; /* elements per row; 0 = input's */

  int64_t tokens;             /* rows T (batch * sequence); 0 is a no-op */
  int32_t n_heads_q, n_heads_k, n_heads_v;          /* >= 0 */
  int32_t head_dim;           /* D: 64 or 128 */

  const float *gamma_q;       /* device fp32 [D]; required when n_heads_q > 0 */
  const float *gamma_k;       /* device fp32 [D]; required when n_heads_k > 0 */
  float eps;                  /* added to mean(x^2); default 1e-6 */

  const void *cos, *sin;      /* device tables, see qknr_cos_layout */
  int32_t cos_dtype;          /* FP32 or BF16 */
  int32_t cos_layout;         /* qknr_cos_layout */
  int64_t cos_rows;           /* table rows; 0 = tokens.  Row of token t: t % cos_rows */
  int32_t rope_style;         /* qknr_rope_style */

  /* Optional device int32.  A kernel whose bounded wait runs out writes a
     nonzero qknr_status here (it never clears it; zero it before the call). */
  int32_t *dev_status;

  /* Launch tuning; 0 = automatic.  See qknr_query(). */
  int32_t ctas_per_sm;        /* persistent CTAs per SM (1..4) */
  int32_t stages;             /* shared-memory ring depth per row group (2..16) */
  int32_t consumer_warps;     /* compute warps per CTA (1..16) */
  int32_t group_warps;        /* warps sharing one row; divides consumer_warps */
  uint32_t flags;             /* QKNR_FLAG_* */
  uint64_t wait_limit_ns;     /* bound on every in-kernel wait; 0 = 2 s */
} qknr_args;

/* What qknr_forward would launch for these arguments. */
typedef struct qknr_launch_info {
  int32_t grid;               /* CTAs (persistent) */
  int32_t block;              /* threads per CTA: consumer warps + 1 producer warp */
  int32_t dyn_smem;           /* dynamic shared memory per CTA, bytes */
  int32_t stages;             /* ring depth per group */
  int32_t ctas_per_sm;
  int32_t consumer_warps;
  int32_t group_warps;        /* consumer warps per row; consumer_warps/group_warps rows in flight */
  int32_t stage_bytes;        /* bytes staged per token row */
  int32_t registers;          /* registers per thread of the chosen kernel */
  int32_t num_sms;
  int32_t prefetch_rows;      /* rows each CTA asks L2 for before its dependency wait (its second
                                 ring fill; 0: none) */
  char kernel[96];            /* kernel variant name */
} qknr_launch_info;

/* Fill *a with defaults: zero pointers and sizes, eps 1e-6, bf16, fp32
   shared-row cos/sin, interleaved, automatic tuning. */
void qknr_args_init(qknr_args *a);

/*
 * Launch the fused QK-RMSNorm + RoPE on `stream` (asynchronous).
 * Returns QKNR_OK after enqueueing, an argument error (nothing launched),
 * or QKNR_ERR_CUDA if the launch failed.  Kernel-side wait timeouts are
 * reported through args->dev_status only.
 *
 * Unless args->flags has QKNR_FLAG_NO_OVERLAP, the kernel is launched with
 * programmatic stream serialization: when the previous operation in the
 * stream is a kernel, this one may launch while that kernel finishes, sets
 * up its shared memory, and then waits for it to complete before it reads
 * or writes any global memory, so stream order holds as with a plain
 * launch.  Before that wait a CTA with many rows only asks L2 to prefetch
 * some of the input rows it will load (Q, K, V segments and table rows
 * inside the buffers given): a prefetch delivers no data to the kernel, and
 * its loads after the wait see the previous kernel's writes.  The prefetch
 * pays when the call overlaps the end of the kernel before it (back-to-back
 * calls, the K call after the Q call); a call that starts cold, after work
 * that does not let it start early, loses about 1 us to it
 * (QKNR_FLAG_NO_PREFETCH skips it; qknr_launch_info.prefetch_rows says
 * whether a launch does it).  Each CTA signals dependents once all of its loads are issued, so
 * a kernel launched after this one the same way (another qknr_forward, for
 * example the K launch after the Q launch) overlaps this one's last rows in
 * the same manner.  A kernel the caller launches after this one with that
 * attribute must itself wait for the grid it depends on before reading the
 * results (cudaGridDependencySynchronize).
 * Thread-safe.
 */
qknr_status qknr_forward(const qknr_args *args, qknr_stream_t stream);

/* Validate *args and describe the launch without launching anything. */
qknr_status qknr_query(const qknr_args *args, qknr_launch_info *info);

/* Short English text of a status code (static storage). */
const char *qknr_status_string(int32_t status);

/* Message of the last error returned on this thread (static per thread). */
const char *qknr_last_error(void);

/*
 * Host-resident activations: the whole call from host buffers
 * ---------------------------------------------------------------
 * For a caller whose activation lives in host memory (a plugin or an
 * offload path that holds the rows on the host; pinned memory makes the
 * copies asynchronous).  qknr_forward_host() streams the token rows through
 * caller-owned device staging buffers in chunks: the host-to-device copy of
 * one chunk, the kernel on the one before and the device-to-host copy of
 * the one before that run at once on three streams, so the call costs about
 * one direction of host-link traffic.  The library still allocates nothing:
 * buffers, copy streams and events all come from the caller.
 *
 * In this call q, k, v, q_out, k_out and v_out of qknr_args are HOST
 * pointers (strides in elements, as for qknr_forward); gamma_q, gamma_k,
 * cos and sin are DEVICE pointers.  Only the columns the operation reads or
 * writes cross the host link: Q and K in and out, and V only when it is
 * copied (v_out set and different from v); in place, V stays where it is.
 * Every row is processed by the same kernel with the same table row as in
 * one qknr_forward() over the whole activation, so the results are the same
 * bits.  A table with cos_rows < tokens (batch broadcast) needs chunk_rows
 * to be a multiple of cos_rows.  With a per-token table and at least four
 * chunks' worth of rows, the first chunks ramp up (chunk_rows/8, /4, /2)
 * and the last ones ramp down, so the copy in of the first chunk and the
 * copy out of the last, which nothing overlaps, stay short; each chunk's
 * table rows are copied in with it.
 */

/* Same type as cudaEvent_t. */
struct CUevent_st;
typedef struct CUevent_st *qknr_event_t;

#define QKNR_HOST_MAX_BUFFERS 4
/* events a plan of n buffers uses */
#define QKNR_HOST_EVENTS(n) (3 * (n) + 2)

typedef struct qknr_host_plan {
  uint32_t abi_version;       /* QKNR_ABI_VERSION */
  int32_t n_buffers;          /* device staging buffers, 1..QKNR_HOST_MAX_BUFFERS; 3 lets copy-in,
                                 kernel and copy-out of consecutive chunks overlap */
  int64_t chunk_rows;         /* token rows per chunk, > 0 */
  /* device staging buffers, 16-byte aligned, each at least
     qknr_host_buffer_bytes() bytes; only the first n_buffers are used */
  void *dev_buffers[QKNR_HOST_MAX_BUFFERS];
  /* the copy streams; either may be the call's stream (then its copies do
     not overlap the kernels) */
  qknr_stream_t h2d_stream, d2h_stream;
  /* caller-created events on the call's device (cudaEventDisableTiming is
     enough); the first QKNR_HOST_EVENTS(n_buffers) are used and re-recorded
     by every call */
  qknr_event_t events[QKNR_HOST_EVENTS(QKNR_HOST_MAX_BUFFERS)];
  /* Optional host copies of the gains and tables.  Each one that is not
     NULL is copied, on h2d_stream before the first chunk, into the device
     buffer that the qknr_args field of the same name points to (gamma: D
     floats; cos, sin: cos_rows table rows, cos_rows = tokens when 0). */
  const void *host_gamma_q, *host_gamma_k, *host_cos, *host_sin;
} qknr_host_plan;

/* Defaults: 3 buffers, 2048-row chunks, everything else zero. */
void qknr_host_plan_init(qknr_host_plan *p);

/* Bytes each device staging buffer needs for these arguments and plan:
   chunk_rows * (n_heads_q + n_heads_k [+ n_heads_v when V is copied]) *
   head_dim * 2. */
qknr_status qknr_host_buffer_bytes(const qknr_args *args, const qknr_host_plan *plan, size_t *bytes);

/*
 * Run the operation on host-resident activations (see above), ordered
 * after the work already on `stream`; once the call returns, `stream`
 * waits for every copy back to the host, so work enqueued on it afterwards
 * (or a synchronisation of it) sees the results.  Nothing is launched when
 * validation fails (argument errors as qknr_forward, plus QKNR_ERR_NULL for
 * a missing buffer or event, QKNR_ERR_SHAPE for chunk_rows / n_buffers out
 * of range or a batch-broadcast table that chunk_rows is not a multiple of,
 * QKNR_ERR_ALIGN for a staging buffer not on 16 bytes, QKNR_ERR_OVERLAP for
 * a host output that partially overlaps a host input).  A CUDA error after
 * the first copy was enqueued returns QKNR_ERR_CUDA; the host outputs are
 * then unspecified.  Thread-safe for calls with distinct plans.
 */
qknr_status qknr_forward_host(const qknr_args *args, const qknr_host_plan *plan, qknr_stream_t stream);

/* sizeof(qknr_host_plan) as compiled into the library. */
size_t qknr_sizeof_host_plan(void);

/* QKNR_ABI_VERSION of the built library. */
int32_t qknr_abi_version(void);

/* sizeof(qknr_args) and sizeof(qknr_launch_info) as compiled into the
   library, so a binding can check its own copy of the layouts. */
size_t qknr_sizeof_args(void);
size_t qknr_sizeof_launch_info(void);

#ifdef __cplusplus
}
#endif

#endif /* QKNR_H_ */
