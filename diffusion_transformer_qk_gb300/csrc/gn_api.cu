// C-ABI launcher of the group-norm + SiLU kernels: validation, piece and
// batch planning, and the launches.  No allocation, no synchronisation.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/qknr_gn.h"
#include "gn_kernel.cuh"
#include "qknr_host.h"

namespace {

using qknr_host::aligned16;
using qknr_host::fail;
using qknr_host::Span;
using qknr_host::span_of;

// Defaults from sweeps on GB300 (VAE decoder maps of 16 MB to 268 MB):
// about 1024 CTAs per launch, and all groups in one launch pair (smaller
// batches that keep the apply pass's re-read in L2 cost more in extra
// launches than they save).
constexpr long long kTargetCtas = 1024;
constexpr long long kMinPiece = 65536;

struct GnPlan {
  qknr::GnParams kp;
  long long spans = 0;          // N * G
  long long piece_len = 0;
  int pieces = 0;
  long long batch_spans = 0;    // spans per launch pair
  size_t workspace = 0;
};

qknr_status plan(const qknr_gn_args* a, GnPlan* pl) {
  if (!a) return fail(QKNR_ERR_NULL, "args is NULL");
  if (a->abi_version != QKNR_ABI_VERSION)
    return fail(QKNR_ERR_ABI, "abi_version %u, library expects %d", a->abi_version, QKNR_ABI_VERSION);
  if (a->dtype != QKNR_BF16 && a->dtype != QKNR_FP16)
    return fail(QKNR_ERR_UNSUPPORTED, "activation dtype must be BF16 or FP16");
  if (a->n <= 0 || a->c <= 0 || a->h <= 0 || a->w <= 0 || a->groups <= 0)
    return fail(QKNR_ERR_SHAPE, "n, c, h, w and groups must be positive");
  if (a->c % a->groups) return fail(QKNR_ERR_SHAPE, "groups must divide channels");
  const long long hw = (long long)a->h * a->w;
  if (hw % 8) return fail(QKNR_ERR_UNSUPPORTED, "H*W must be a multiple of 8");
  const long long L = (long long)(a->c / a->groups) * hw;
  if (L >= (1ll << 31)) return fail(QKNR_ERR_UNSUPPORTED, "a group of 2^31 or more elements");
  if (!(a->eps >= 0.0f)) return fail(QKNR_ERR_SHAPE, "eps must be >= 0");
  if (a->piece_elems < 0 || a->piece_elems % 8) return fail(QKNR_ERR_SHAPE, "piece_elems must be a multiple of 8");
  if (a->l2_batch_bytes < -1) return fail(QKNR_ERR_SHAPE, "l2_batch_bytes must be >= -1");

  pl->spans = (long long)a->n * a->groups;
  long long piece = a->piece_elems;
  if (piece == 0) {
    const long long want_p = (kTargetCtas + pl->spans - 1) / pl->spans;
    piece = (L + want_p - 1) / want_p;
    if (piece < kMinPiece) piece = kMinPiece;
    piece = (piece + 7) / 8 * 8;
  }
  if (piece > L) piece = (L + 7) / 8 * 8;
  const long long P = (L + piece - 1) / piece;
  if (P > 65535) return fail(QKNR_ERR_UNSUPPORTED, "more than 65535 pieces per group");
  pl->piece_len = piece;
  pl->pieces = static_cast<int>(P);
  pl->workspace = static_cast<size_t>(pl->spans * (P + 1) * 2 * sizeof(double));
  const long long span_bytes = L * 2;
  const long long batch_bytes = a->l2_batch_bytes;
  long long bs = batch_bytes <= 0 ? pl->spans : batch_bytes / span_bytes;
  if (bs < 1) bs = 1;
  if (bs > pl->spans) bs = pl->spans;
  if (bs > 65535) bs = 65535;
  pl->batch_spans = bs;

  qknr::GnParams& kp = pl->kp;
  memset(&kp, 0, sizeof(kp));
  kp.x = static_cast<const char*>(a->x);
  kp.out = static_cast<char*>(a->out ? a->out : const_cast<void*>(a->x));
  kp.gamma = a->gamma;
  kp.beta = a->beta;
  kp.partial = static_cast<double*>(a->workspace);
  kp.span_len = L;
  kp.hw = hw;
  kp.piece_len = piece;
  kp.channels = a->c;
  kp.groups = a->groups;
  kp.group_channels = a->c / a->groups;
  kp.pieces = pl->pieces;
  kp.eps = a->eps;
  return QKNR_OK;
}

qknr_status check_buffers(const qknr_gn_args* a, const GnPlan& pl) {
  if (!a->x || !a->gamma || !a->beta) return fail(QKNR_ERR_NULL, "x, gamma and beta are required");
  if (!a->workspace) return fail(QKNR_ERR_NULL, "workspace is required (qknr_gn_workspace_bytes)");
  if (a->workspace_bytes < pl.workspace)
    return fail(QKNR_ERR_SHAPE, "workspace of %zu bytes, %zu needed", a->workspace_bytes, pl.workspace);
  const void* out = a->out ? a->out : a->x;
  if (!aligned16(a->x) || !aligned16(out) || !aligned16(a->workspace) ||
      (reinterpret_cast<uintptr_t>(a->gamma) & 3u) || (reinterpret_cast<uintptr_t>(a->beta) & 3u))
    return fail(QKNR_ERR_ALIGN, "x / out / workspace not 16-byte aligned, or gamma / beta not 4-byte aligned");
  const long long total = pl.spans * pl.kp.span_len * 2;
  const Span sx = span_of(a->x, 1, 0, total), so = span_of(out, 1, 0, total);
  const Span sw = span_of(a->workspace, 1, 0, static_cast<long long>(pl.workspace));
  const Span sg = span_of(a->gamma, 1, 0, (long long)a->c * 4), sb = span_of(a->beta, 1, 0, (long long)a->c * 4);
  if (out != a->x && (qknr_host::overlaps(so, sx) || qknr_host::overlaps(so, sg) || qknr_host::overlaps(so, sb) ||
                      qknr_host::overlaps(so, sw)))
    return fail(QKNR_ERR_OVERLAP, "out overlaps an input without being in place");
  if (qknr_host::overlaps(sw, sx) || qknr_host::overlaps(sw, sg) || qknr_host::overlaps(sw, sb))
    return fail(QKNR_ERR_OVERLAP, "workspace overlaps an input");
  return QKNR_OK;
}

}  // namespace

extern "C" {

void qknr_gn_args_init(qknr_gn_args* a) {
  if (!a) return;
  memset(a, 0, sizeof(*a));
  a->abi_version = QKNR_ABI_VERSION;
  a->dtype = QKNR_BF16;
  a->eps = 1e-6f;
}

qknr_status qknr_gn_workspace_bytes(const qknr_gn_args* args, size_t* bytes) {
  if (!bytes) return fail(QKNR_ERR_NULL, "bytes is NULL");
  GnPlan pl;
  qknr_status st = plan(args, &pl);
  if (st != QKNR_OK) return st;
  *bytes = pl.workspace;
  return QKNR_OK;
}

qknr_status qknr_gn_silu_forward(const qknr_gn_args* args, qknr_stream_t stream) {
  GnPlan pl;
  qknr_status st = plan(args, &pl);
  if (st != QKNR_OK) return st;
  st = check_buffers(args, pl);
  if (st != QKNR_OK) return st;
  const bool bf16 = args->dtype == QKNR_BF16;
  const void* stats = bf16 ? reinterpret_cast<const void*>(&qknr::gn_stats_kernel<__nv_bfloat16>)
                           : reinterpret_cast<const void*>(&qknr::gn_stats_kernel<__half>);
  const void* apply = bf16 ? reinterpret_cast<const void*>(&qknr::gn_apply_kernel<__nv_bfloat16>)
                           : reinterpret_cast<const void*>(&qknr::gn_apply_kernel<__half>);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (long long s0 = 0; s0 < pl.spans; s0 += pl.batch_spans) {
    qknr::GnParams kp = pl.kp;
    kp.span0 = static_cast<int>(s0);
    const long long nb = pl.spans - s0 < pl.batch_spans ? pl.spans - s0 : pl.batch_spans;
    const dim3 grid(static_cast<unsigned>(pl.pieces), static_cast<unsigned>(nb));
    void* kargs[] = {&kp};
    cudaError_t e = cudaLaunchKernel(stats, grid, dim3(qknr::kGnThreads), kargs, 0, s);
    if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaLaunchKernel(group norm statistics)");
    e = cudaLaunchKernel(apply, grid, dim3(qknr::kGnThreads), kargs, 0, s);
    if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaLaunchKernel(group norm apply)");
  }
  return QKNR_OK;
}

size_t qknr_gn_sizeof_args(void) { return sizeof(qknr_gn_args); }

}  // extern "C"

// ---------------------------------------------------------------------------
// The same call for callers that may not allocate device memory.
//
// Some callers cannot hand the library a workspace: code that runs inside a
// host framework's enqueue step with no allocator of its own, a plugin
// whose workspace size had to be fixed before the shapes were known, or a
// runtime that keeps a fixed device-memory budget and forbids cudaMalloc
// (which also synchronises the device) on its execution path.  For them the
// statistics go to this fixed array, which every device that loads the
// library holds until the process exits.

namespace {

// Room for the per-piece sums of QKNR_GN_NOALLOC_SCRATCH_BYTES / 16
// (sample, group, piece) records.
static __device__ __align__(256) double g_gn_noalloc_scratch[QKNR_GN_NOALLOC_SCRATCH_BYTES / sizeof(double)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached.
qknr_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(QKNR_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gn_noalloc_scratch);
    if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaGetSymbolAddress(group-norm scratch)");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return QKNR_OK;
}

}  // namespace

extern "C" qknr_status qknr_gn_silu_forward_noalloc(const qknr_gn_args* args, qknr_stream_t stream) {
  if (!args) return fail(QKNR_ERR_NULL, "args is NULL");
  qknr_gn_args a = *args;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  size_t need = 0;
  qknr_status st = qknr_gn_workspace_bytes(&a, &need);
  if (st != QKNR_OK) return st;
  if (need > QKNR_GN_NOALLOC_SCRATCH_BYTES)
    return fail(QKNR_ERR_UNSUPPORTED,
                "this shape needs %zu bytes of statistics scratch; the no-allocation entry point has %d "
                "(use fewer pieces per group, or qknr_gn_silu_forward with a workspace)",
                need, QKNR_GN_NOALLOC_SCRATCH_BYTES);
  // argument errors come back before the first CUDA call (the address lookup)
  if (!a.x || !a.gamma || !a.beta) return fail(QKNR_ERR_NULL, "x, gamma and beta are required");
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != QKNR_OK) return st;
  a.workspace = scratch;
  a.workspace_bytes = QKNR_GN_NOALLOC_SCRATCH_BYTES;
  return qknr_gn_silu_forward(&a, stream);
}
