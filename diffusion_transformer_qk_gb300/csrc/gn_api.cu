// C-ABI launcher of the group-norm + SiLU kernels: validation, the choice
// between the cluster, fused and two-pass paths, the cluster split, piece
// and batch planning, and the launches.  No allocation, no
// synchronisation.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/qknr_gn.h"
#include "gn_cluster.cuh"
#include "gn_kernel.cuh"
#include "qknr_host.h"

namespace {

using qknr_host::aligned16;
using qknr_host::fail;
using qknr_host::Span;
using qknr_host::span_of;

// Two-pass defaults from sweeps on GB300 (VAE decoder maps of 16 MB to
// 268 MB): about 1024 CTAs per launch, and all groups in one launch pair
// (smaller batches that keep the apply pass's re-read in L2 cost more in
// extra launches than they save).
constexpr long long kTargetCtas = 1024;
constexpr long long kMinPiece = 65536;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

struct GnPlan {
  long long spans = 0;          // N * G
  long long L = 0;              // elements per span
  // two-pass path
  qknr::GnParams kp;
  long long piece_len = 0;
  int pieces = 0;
  long long batch_spans = 0;    // spans per launch pair
  size_t ws_two = 0;
  // fused path (sizes that do not depend on the device)
  bool fused_shape = false;     // chunk count in range
  unsigned f_pieces = 0;        // P = ceil(L / kGnfChunk)
  size_t f_records = 0;         // bytes of the [spans][P + 1] 16-byte records
  size_t ws_fused = 0;
  bool want_fused = false;      // AUTO without two-pass tuning, or FUSED
  // cluster path (sizes that do not depend on the device)
  bool cluster_shape = false;   // a group fits the shared memory of a cluster (200 KB parts)
  bool cluster_auto = false;    // ... with parts of at most 32 KB
  bool want_cluster = false;    // AUTO without two-pass tuning on such a shape, or CLUSTER
  size_t workspace = 0;         // what qknr_gn_workspace_bytes reports
};

// The cluster path's split of a group of L elements over c CTAs (a power
// of two up to kGncMaxCluster): parts of at most 32 KB where a cluster can
// hold the group so (the automatic choice takes the cluster path only
// then), else, when asked for, of at most 200 KB; then, while the grid
// would have fewer than two CTAs per SM and parts stay at 4 KB or more,
// twice as many CTAs per group.  Sweeps on GB300 (flushed calls): groups of
// 32 KB to 512 KB ran 15-25 % faster than on the fused path with parts of
// 8-32 KB; groups of 1 MB tied it and of 2 MB took 60 % longer (few
// clusters of 16 fit at once).
constexpr long long kGncSmallPartBytes = 32 * 1024;
constexpr long long kGncMaxPartBytes = 200 * 1024;
constexpr long long kGncMinPartBytes = 4 * 1024;

long long cluster_part(long long L, int c) { return ((L + c - 1) / c + 7) / 8 * 8; }

// smallest c whose parts fit `cap` bytes, or 0
int cluster_fit(long long L, long long cap) {
  for (int c = 1; c <= qknr::kGncMaxCluster; c *= 2)
    if (cluster_part(L, c) * 2 <= cap) return c;
  return 0;
}

void cluster_split(long long L, long long spans, int num_sms, bool allow_large, int* cluster, long long* part_len) {
  int c = cluster_fit(L, kGncSmallPartBytes);
  if (c == 0 && allow_large) c = cluster_fit(L, kGncMaxPartBytes);
  while (c > 0 && c < qknr::kGncMaxCluster && spans * c < 2ll * num_sms &&
         cluster_part(L, 2 * c) * 2 >= kGncMinPartBytes)
    c *= 2;
  *cluster = c;
  *part_len = c > 0 ? cluster_part(L, c) : 0;
}

qknr_status plan(const qknr_gn_args* a, GnPlan* pl) {
  if (!a) return fail(QKNR_ERR_NULL, "args is NULL");
  if (a->abi_version != QKNR_ABI_VERSION)
    return fail(QKNR_ERR_ABI, "abi_version %u, library expects %d", a->abi_version, QKNR_ABI_VERSION);
  if (a->dtype != QKNR_BF16 && a->dtype != QKNR_FP16)
    return fail(QKNR_ERR_UNSUPPORTED, "activation dtype must be BF16 or FP16");
  if (a->mode != QKNR_GN_AUTO && a->mode != QKNR_GN_FUSED && a->mode != QKNR_GN_TWO_PASS &&
      a->mode != QKNR_GN_CLUSTER)
    return fail(QKNR_ERR_UNSUPPORTED, "unknown mode %d", a->mode);
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
  pl->L = L;

  // ---- two-pass path
  long long piece = a->piece_elems;
  if (piece == 0) {
    const long long want_p = (kTargetCtas + pl->spans - 1) / pl->spans;
    piece = (L + want_p - 1) / want_p;
    if (piece < kMinPiece) piece = kMinPiece;
    piece = (piece + 7) / 8 * 8;
  }
  if (piece > L) piece = (L + 7) / 8 * 8;
  const long long P = (L + piece - 1) / piece;
  const bool two_ok = P <= 65535;
  pl->piece_len = piece;
  pl->pieces = static_cast<int>(two_ok ? P : 0);
  pl->ws_two = static_cast<size_t>(pl->spans * (P + 1) * 2 * sizeof(double));
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
  kp.rec = static_cast<unsigned long long*>(a->workspace);
  kp.span_len = L;
  kp.hw = hw;
  kp.piece_len = piece;
  kp.channels = a->c;
  kp.groups = a->groups;
  kp.group_channels = a->c / a->groups;
  kp.pieces = pl->pieces;
  kp.eps = a->eps;
  kp.status = a->dev_status;

  // ---- fused path
  const long long fP = (L + qknr::kGnfChunk - 1) / qknr::kGnfChunk;
  pl->fused_shape = pl->spans * fP < (1ll << 31);
  pl->f_pieces = static_cast<unsigned>(fP);
  pl->f_records = static_cast<size_t>(pl->spans * (fP + 1) * 2 * sizeof(double));
  pl->ws_fused = pl->f_records + 16;   // + the abort word

  // ---- cluster path (the split itself depends on the device's SM count)
  const bool grid_ok = pl->spans <= 0x7fffffffll / qknr::kGncMaxCluster;
  pl->cluster_shape = grid_ok && cluster_fit(L, kGncMaxPartBytes) > 0;
  pl->cluster_auto = grid_ok && cluster_fit(L, kGncSmallPartBytes) > 0;

  const bool tuned = a->piece_elems != 0 || a->l2_batch_bytes != 0;
  pl->want_cluster = a->mode == QKNR_GN_CLUSTER || (a->mode == QKNR_GN_AUTO && !tuned && pl->cluster_auto);
  pl->want_fused = a->mode == QKNR_GN_FUSED || (a->mode == QKNR_GN_AUTO && !tuned);
  if (a->mode == QKNR_GN_CLUSTER) {
    if (!pl->cluster_shape)
      return fail(QKNR_ERR_UNSUPPORTED, "a group of %lld elements does not fit a cluster of %d CTAs", L,
                  qknr::kGncMaxCluster);
    pl->want_fused = false;
    pl->workspace = 0;                   // the cluster path keeps its statistics on chip
    return QKNR_OK;
  }
  if (a->mode == QKNR_GN_FUSED) {
    if (!pl->fused_shape) return fail(QKNR_ERR_UNSUPPORTED, "2^31 or more pieces in all for the fused path");
    pl->workspace = pl->ws_fused;
  } else if (pl->want_fused && pl->fused_shape) {
    if (!two_ok) {
      pl->workspace = pl->ws_fused;   // only the fused path could run this shape
    } else {
      pl->workspace = pl->ws_two > pl->ws_fused ? pl->ws_two : pl->ws_fused;
    }
  } else {
    pl->want_fused = false;
    if (!two_ok) return fail(QKNR_ERR_UNSUPPORTED, "more than 65535 pieces per group");
    pl->workspace = pl->ws_two;
  }
  return QKNR_OK;
}

// The fused launch on the current device, or why there is none.
struct FusedLaunch {
  bool ok = false;
  const void* fn = nullptr;
  int grid = 0;
  int per_cta = 0;            // most pieces of one group a CTA holds
  int regs = 0;
  int num_sms = 0;
  char why[160] = "";
};

qknr_status fused_launch(const qknr_gn_args* a, const GnPlan& pl, FusedLaunch* fl) {
  fl->fn = a->dtype == QKNR_BF16 ? reinterpret_cast<const void*>(&qknr::gn_fused_kernel<__nv_bfloat16>)
                                 : reinterpret_cast<const void*>(&qknr::gn_fused_kernel<__half>);
  if (!pl.fused_shape) {
    snprintf(fl->why, sizeof(fl->why), "2^31 or more pieces in all");
    return QKNR_OK;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaGetDevice");
  qknr_host::DeviceInfo di;
  qknr_status st = qknr_host::device_info(dev, &di);
  if (st != QKNR_OK) return st;
  fl->num_sms = di.num_sms;
  if (!di.cooperative) {
    snprintf(fl->why, sizeof(fl->why), "the device has no cooperative launch");
    return QKNR_OK;
  }
  if (di.smem_optin < qknr::kGnfSmemBytes) {
    snprintf(fl->why, sizeof(fl->why), "%d bytes of shared memory per block, %d needed", di.smem_optin,
             qknr::kGnfSmemBytes);
    return QKNR_OK;
  }
  st = qknr_host::configure_kernel(fl->fn, dev, di, &fl->regs);
  if (st != QKNR_OK) return st;
  const long long chunks = pl.spans * static_cast<long long>(pl.f_pieces);
  const long long G = chunks < di.num_sms ? chunks : di.num_sms;      // one CTA per SM
  // a CTA holds at most ceil(P / G) pieces of a group; at most kGnfSlots
  // keeps every wait finite
  const long long per_cta = (pl.f_pieces + G - 1) / G;
  if (per_cta > qknr::kGnfSlots) {
    snprintf(fl->why, sizeof(fl->why), "a group of %u pieces needs %lld per CTA on %lld CTAs (at most %d)",
             pl.f_pieces, per_cta, G, qknr::kGnfSlots);
    return QKNR_OK;
  }
  fl->grid = static_cast<int>(G);
  fl->per_cta = static_cast<int>(per_cta);
  fl->ok = true;
  return QKNR_OK;
}

// The cluster launch on the current device, or why there is none.
struct ClusterLaunch {
  bool ok = false;
  const void* fn = nullptr;
  int cluster = 0;            // CTAs per cluster (per group of a sample)
  long long part_len = 0;     // elements per CTA
  int threads = 0;            // per CTA
  int grid = 0;
  int smem = 0;
  int regs = 0;
  int num_sms = 0;
  int max_clusters = 0;       // clusters of this launch resident at once
  char why[160] = "";
};

// The automatic choice takes the cluster path only when every group's
// cluster fits on the GPU at once: a CTA loads, merges and writes its part
// one step after the other, so a second wave of clusters leaves DRAM idle
// in between (8 x 512 x 128 x 128, 256 groups of 512 KB in waves of 33
// clusters: 76.9 us flushed, where the fused path reads at the copy rate).
qknr_status one_wave(const qknr_gn_args* a, const GnPlan& pl, ClusterLaunch* cl) {
  if (a->mode == QKNR_GN_AUTO && pl.spans > cl->max_clusters) {
    cl->ok = false;
    snprintf(cl->why, sizeof(cl->why), "%lld groups, %d clusters of %d CTAs at once", pl.spans, cl->max_clusters,
             cl->cluster);
  }
  return QKNR_OK;
}

qknr_status cluster_launch(const qknr_gn_args* a, const GnPlan& pl, ClusterLaunch* cl) {
  cl->fn = a->dtype == QKNR_BF16 ? reinterpret_cast<const void*>(&qknr::gn_cluster_kernel<__nv_bfloat16, 256>)
                                 : reinterpret_cast<const void*>(&qknr::gn_cluster_kernel<__half, 256>);
  cl->threads = 256;
  if (!pl.cluster_shape) {
    snprintf(cl->why, sizeof(cl->why), "a group does not fit a cluster");
    return QKNR_OK;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaGetDevice");
  qknr_host::DeviceInfo di;
  qknr_status st = qknr_host::device_info(dev, &di);
  if (st != QKNR_OK) return st;
  cl->num_sms = di.num_sms;
  int cluster_launch = 0;
  e = cudaDeviceGetAttribute(&cluster_launch, cudaDevAttrClusterLaunch, dev);
  if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaDeviceGetAttribute(ClusterLaunch)");
  if (!cluster_launch) {
    snprintf(cl->why, sizeof(cl->why), "the device has no cluster launch");
    return QKNR_OK;
  }
  cluster_split(pl.L, pl.spans, di.num_sms, a->mode == QKNR_GN_CLUSTER, &cl->cluster, &cl->part_len);
  cl->smem = static_cast<int>(qknr::kGncOffData + cl->part_len * 2);
  if (di.smem_optin < cl->smem) {
    snprintf(cl->why, sizeof(cl->why), "%d bytes of shared memory per block, %d needed", di.smem_optin, cl->smem);
    return QKNR_OK;
  }
  st = qknr_host::configure_kernel(cl->fn, dev, di, &cl->regs);
  if (st != QKNR_OK) return st;
  // clusters of this size and shared memory that fit at once, asked once
  // per kernel, device, size and shared memory
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, int>, int> resident;
  const auto key = std::make_tuple(cl->fn, dev, cl->cluster, cl->smem);   // fn fixes the threads
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = resident.find(key);
    if (it != resident.end()) {
      cl->max_clusters = it->second;
      if (it->second < 1) {
        snprintf(cl->why, sizeof(cl->why), "no cluster of %d CTAs with %d bytes each fits", cl->cluster, cl->smem);
        return QKNR_OK;
      }
      cl->grid = static_cast<int>(pl.spans * cl->cluster);
      cl->ok = true;
      return one_wave(a, pl, cl);
    }
  }
  if (cl->cluster > 8) {
    e = cudaFuncSetAttribute(cl->fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaFuncSetAttribute(NonPortableClusterSizeAllowed)");
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cl->cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(pl.spans * cl->cluster));
  cfg.blockDim = dim3(static_cast<unsigned>(cl->threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(cl->smem);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, cl->fn, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();                  // a configuration the device cannot place: not sticky
    n = 0;
  }
  {
    std::lock_guard<std::mutex> lk(mu);
    resident[key] = n;
  }
  if (n < 1) {
    snprintf(cl->why, sizeof(cl->why), "no cluster of %d CTAs with %d bytes each fits", cl->cluster, cl->smem);
    return QKNR_OK;
  }
  cl->max_clusters = n;
  cl->grid = static_cast<int>(pl.spans * cl->cluster);
  cl->ok = true;
  return one_wave(a, pl, cl);
}

// Resolve the path: *use_fused, with fl filled when it is true.
qknr_status choose(const qknr_gn_args* a, const GnPlan& pl, FusedLaunch* fl, bool* use_fused) {
  *use_fused = false;
  if (!pl.want_fused) return QKNR_OK;
  qknr_status st = fused_launch(a, pl, fl);
  if (st != QKNR_OK) return st;
  if (fl->ok) {
    *use_fused = true;
    return QKNR_OK;
  }
  if (a->mode == QKNR_GN_FUSED) return fail(QKNR_ERR_UNSUPPORTED, "fused group norm: %s", fl->why);
  if (pl.pieces == 0) return fail(QKNR_ERR_UNSUPPORTED, "more than 65535 pieces per group (and fused: %s)", fl->why);
  return QKNR_OK;
}

qknr_status check_buffers(const qknr_gn_args* a, const GnPlan& pl) {
  if (!a->x || !a->gamma || !a->beta) return fail(QKNR_ERR_NULL, "x, gamma and beta are required");
  if (!a->workspace && pl.workspace > 0)
    return fail(QKNR_ERR_NULL, "workspace is required (qknr_gn_workspace_bytes)");
  if (a->workspace_bytes < pl.workspace)
    return fail(QKNR_ERR_SHAPE, "workspace of %zu bytes, %zu needed", a->workspace_bytes, pl.workspace);
  const void* out = a->out ? a->out : a->x;
  if (!aligned16(a->x) || !aligned16(out) || !aligned16(a->workspace) ||
      (reinterpret_cast<uintptr_t>(a->gamma) & 3u) || (reinterpret_cast<uintptr_t>(a->beta) & 3u) ||
      (reinterpret_cast<uintptr_t>(a->dev_status) & 3u))
    return fail(QKNR_ERR_ALIGN,
                "x / out / workspace not 16-byte aligned, or gamma / beta / dev_status not 4-byte aligned");
  const long long total = pl.spans * pl.L * 2;
  const Span sx = span_of(a->x, 1, 0, total), so = span_of(out, 1, 0, total);
  const Span sw = span_of(a->workspace, 1, 0, static_cast<long long>(pl.workspace));
  const Span sg = span_of(a->gamma, 1, 0, (long long)a->c * 4), sb = span_of(a->beta, 1, 0, (long long)a->c * 4);
  if (out != a->x && (qknr_host::overlaps(so, sx) || qknr_host::overlaps(so, sg) || qknr_host::overlaps(so, sb) ||
                      qknr_host::overlaps(so, sw)))
    return fail(QKNR_ERR_OVERLAP, "out overlaps an input without being in place");
  if (pl.workspace > 0 &&
      (qknr_host::overlaps(sw, sx) || qknr_host::overlaps(sw, sg) || qknr_host::overlaps(sw, sb)))
    return fail(QKNR_ERR_OVERLAP, "workspace overlaps an input");
  return QKNR_OK;
}

// Address spans of a call's buffers, which checked builds test every access
// against: x and out (N*C*H*W elements), the part of the workspace the call
// uses, gamma and beta.
struct GnSpans {
  qknr::MemSpan x, out, ws, gamma, beta;
};

GnSpans spans_of(const qknr_gn_args* a, const GnPlan& pl) {
  const long long total = pl.spans * pl.L * 2;
  const void* out = a->out ? a->out : a->x;
  auto ms = [](Span x) { return qknr::MemSpan{x.lo, x.hi}; };
  return {ms(span_of(a->x, 1, 0, total)), ms(span_of(out, 1, 0, total)),
          ms(span_of(a->workspace, 1, 0, static_cast<long long>(pl.workspace))),
          ms(span_of(a->gamma, 1, 0, (long long)a->c * 4)), ms(span_of(a->beta, 1, 0, (long long)a->c * 4))};
}

// The tag of calls made while the stream is being captured into a CUDA
// graph: a replay reuses its launch's parameters, so the captured call
// clears the records first (a memset node) and uses this fixed tag.
constexpr unsigned kCaptureTag = 1u;

// A per-call record tag: a bijective 32-bit mix of a process-wide call
// counter (no tag repeats within 2^32 calls; tags do not look like small
// integers or zeros left in a reused workspace), never 0 (the two-pass tag)
// and never kCaptureTag.
unsigned next_tag() {
  static std::atomic<unsigned> counter{0};
  while (true) {
    unsigned x = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
    x *= 0x9E3779B1u;
    x ^= x >> 16;
    x *= 0x85EBCA6Bu;
    x ^= x >> 13;
    if (x != 0u && x != kCaptureTag) return x;
  }
}

// *too_large: the cooperative launch did not fit the SMs this context may
// use (e.g. under MPS); in QKNR_GN_AUTO the caller then takes the two-pass
// path, whose workspace the auto size already covers.
qknr_status launch_fused(const qknr_gn_args* a, const GnPlan& pl, const FusedLaunch& fl, cudaStream_t s,
                         bool* too_large) {
  *too_large = false;
  char* ws = static_cast<char*>(a->workspace);
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &capture);
  if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaStreamIsCapturing");
  unsigned tag = 0;
  if (capture == cudaStreamCaptureStatusActive) {
    // every replay starts from cleared records and abort word
    e = cudaMemsetAsync(ws, 0, pl.f_records + 16, s);
    if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaMemsetAsync(group norm records)");
    tag = kCaptureTag;
  } else {
    tag = next_tag();
  }
  qknr::GnFusedParams fp;
  memset(&fp, 0, sizeof(fp));
  fp.x = static_cast<const char*>(a->x);
  fp.out = static_cast<char*>(a->out ? a->out : const_cast<void*>(a->x));
  fp.gamma = a->gamma;
  fp.beta = a->beta;
  fp.rec = reinterpret_cast<unsigned long long*>(ws);
  fp.abort_word = reinterpret_cast<unsigned*>(ws + pl.f_records);
  fp.status = a->dev_status;
  fp.span_len = pl.L;
  fp.hw = (long long)a->h * a->w;
  fp.pieces = pl.f_pieces;
  fp.total_chunks = static_cast<unsigned>(pl.spans * static_cast<long long>(pl.f_pieces));
  fp.groups = a->groups;
  fp.group_channels = a->c / a->groups;
  fp.channels = a->c;
  fp.tag = tag;
  fp.flags = a->flags & (qknr::kGnfFlagStallLoads | qknr::kGnfFlagStallRecords);
  fp.wait_limit_ns = a->wait_limit_ns ? a->wait_limit_ns : kDefaultWaitNs;
  fp.eps = a->eps;
  const GnSpans sp = spans_of(a, pl);
  fp.sp_x = sp.x;
  fp.sp_out = sp.out;
  fp.sp_ws = sp.ws;
  fp.sp_gamma = sp.gamma;
  fp.sp_beta = sp.beta;
  void* kargs[] = {&fp};
  e = cudaLaunchCooperativeKernel(fl.fn, dim3(fl.grid), dim3(qknr::kGnfThreads), kargs,
                                              static_cast<size_t>(qknr::kGnfSmemBytes), s);
  if (e == cudaErrorCooperativeLaunchTooLarge && a->mode == QKNR_GN_AUTO && pl.pieces > 0) {
    (void)cudaGetLastError();                  // a launch-configuration error: not sticky
    *too_large = true;
    return QKNR_OK;
  }
  if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaLaunchCooperativeKernel(fused group norm)");
  return QKNR_OK;
}

qknr_status launch_cluster(const qknr_gn_args* a, const GnPlan& pl, const ClusterLaunch& cl, cudaStream_t s) {
  qknr::GnClusterParams cp;
  memset(&cp, 0, sizeof(cp));
  cp.x = static_cast<const char*>(a->x);
  cp.out = static_cast<char*>(a->out ? a->out : const_cast<void*>(a->x));
  cp.gamma = a->gamma;
  cp.beta = a->beta;
  cp.status = a->dev_status;
  cp.span_len = pl.L;
  cp.hw = (long long)a->h * a->w;
  cp.part_len = cl.part_len;
  cp.groups = a->groups;
  cp.group_channels = a->c / a->groups;
  cp.flags = a->flags & qknr::kGnfFlagStallLoads;
  cp.smem_bytes = static_cast<unsigned>(cl.smem);
  cp.wait_limit_ns = a->wait_limit_ns ? a->wait_limit_ns : kDefaultWaitNs;
  cp.eps = a->eps;
  const GnSpans sp = spans_of(a, pl);
  cp.sp_x = sp.x;
  cp.sp_out = sp.out;
  cp.sp_gamma = sp.gamma;
  cp.sp_beta = sp.beta;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cl.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(cl.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(cl.threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(cl.smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* kargs[] = {&cp};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, cl.fn, kargs);
  if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaLaunchKernelExC(cluster group norm)");
  return QKNR_OK;
}

qknr_status launch_two_pass(const qknr_gn_args* a, const GnPlan& pl, cudaStream_t s) {
  const bool bf16 = a->dtype == QKNR_BF16;
  const void* stats = bf16 ? reinterpret_cast<const void*>(&qknr::gn_stats_kernel<__nv_bfloat16>)
                           : reinterpret_cast<const void*>(&qknr::gn_stats_kernel<__half>);
  const void* apply = bf16 ? reinterpret_cast<const void*>(&qknr::gn_apply_kernel<__nv_bfloat16>)
                           : reinterpret_cast<const void*>(&qknr::gn_apply_kernel<__half>);
  const GnSpans sp = spans_of(a, pl);
  for (long long s0 = 0; s0 < pl.spans; s0 += pl.batch_spans) {
    qknr::GnParams kp = pl.kp;
    kp.span0 = static_cast<int>(s0);
    kp.sp_x = sp.x;
    kp.sp_out = sp.out;
    kp.sp_ws = sp.ws;
    kp.sp_gamma = sp.gamma;
    kp.sp_beta = sp.beta;
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

}  // namespace

extern "C" {

void qknr_gn_args_init(qknr_gn_args* a) {
  if (!a) return;
  memset(a, 0, sizeof(*a));
  a->abi_version = QKNR_ABI_VERSION;
  a->dtype = QKNR_BF16;
  a->eps = 1e-6f;
  a->mode = QKNR_GN_AUTO;
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
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (pl.want_cluster) {
    ClusterLaunch cl;
    st = cluster_launch(args, pl, &cl);
    if (st != QKNR_OK) return st;
    if (cl.ok) return launch_cluster(args, pl, cl, s);
    if (args->mode == QKNR_GN_CLUSTER) return fail(QKNR_ERR_UNSUPPORTED, "cluster group norm: %s", cl.why);
  }
  FusedLaunch fl;
  bool fused = false;
  st = choose(args, pl, &fl, &fused);
  if (st != QKNR_OK) return st;
  if (fused) {
    bool too_large = false;
    st = launch_fused(args, pl, fl, s, &too_large);
    if (st != QKNR_OK || !too_large) return st;
  }
  return launch_two_pass(args, pl, s);
}

qknr_status qknr_gn_query(const qknr_gn_args* args, qknr_launch_info* info) {
  if (!info) return fail(QKNR_ERR_NULL, "info is NULL");
  memset(info, 0, sizeof(*info));
  GnPlan pl;
  qknr_status st = plan(args, &pl);
  if (st != QKNR_OK) return st;
  const char* dt = args->dtype == QKNR_BF16 ? "bf16" : "fp16";
  if (pl.want_cluster) {
    ClusterLaunch cl;
    st = cluster_launch(args, pl, &cl);
    if (st != QKNR_OK) return st;
    if (cl.ok) {
      info->grid = cl.grid;
      info->block = cl.threads;
      info->dyn_smem = cl.smem;
      info->stages = 1;
      info->ctas_per_sm = 0;
      info->consumer_warps = cl.threads / 32;
      info->stage_bytes = static_cast<int32_t>(cl.part_len * 2);
      info->registers = cl.regs;
      info->num_sms = cl.num_sms;
      snprintf(info->kernel, sizeof(info->kernel), "gn_cluster<%s>, clusters of %d CTAs, %lld elements each, %d resident",
               dt, cl.cluster, cl.part_len, cl.max_clusters);
      return QKNR_OK;
    }
    if (args->mode == QKNR_GN_CLUSTER) return fail(QKNR_ERR_UNSUPPORTED, "cluster group norm: %s", cl.why);
  }
  FusedLaunch fl;
  bool fused = false;
  st = choose(args, pl, &fl, &fused);
  if (st != QKNR_OK) return st;
  if (fused) {
    info->grid = fl.grid;
    info->block = qknr::kGnfThreads;
    info->dyn_smem = qknr::kGnfSmemBytes;
    info->stages = qknr::kGnfSlots;
    info->ctas_per_sm = 1;
    info->consumer_warps = qknr::kGnfStatsWarps + qknr::kGnfApplyWarps;
    info->stage_bytes = qknr::kGnfChunkBytes;
    info->registers = fl.regs;
    info->num_sms = fl.num_sms;
    snprintf(info->kernel, sizeof(info->kernel), "gn_fused<%s>, %u pieces per group, %d per CTA", dt,
             pl.f_pieces, fl.per_cta);
  } else {
    const long long nb = pl.batch_spans;
    info->grid = static_cast<int32_t>(pl.pieces * nb);
    info->block = qknr::kGnThreads;
    info->stage_bytes = static_cast<int32_t>(pl.piece_len * 2);
    snprintf(info->kernel, sizeof(info->kernel), "gn_stats+gn_apply<%s> x%lld, %d pieces per group", dt,
             (pl.spans + nb - 1) / nb, pl.pieces);
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
