// C-ABI launcher of the fused DiT QK-RMSNorm + RoPE kernels: argument
// validation, launch planning (persistent grid, stage ring depth, shared
// memory) and the launch itself.  No allocation, no synchronisation.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <unordered_map>
#include <utility>

#include "../../include/qknr.h"
#include "qknr_internal.h"
#include "qknr_host.h"

namespace qknr_host {

thread_local char g_err[512] = "";

qknr_status fail(qknr_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

qknr_status cuda_fail(cudaError_t e, const char* what) {
  return fail(QKNR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
std::mutex g_mu;
std::unordered_map<int, DeviceInfo> g_dev;
std::map<std::pair<const void*, int>, int> g_configured;   // (kernel, device) -> registers per thread
}  // namespace

qknr_status device_info(int dev, DeviceInfo* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_dev.find(dev);
  if (it != g_dev.end()) {
    *out = it->second;
    return QKNR_OK;
  }
  DeviceInfo d;
  cudaError_t e;
  if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
  if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
      cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(MaxSharedMemoryPerBlockOptin)");
  if ((e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
      cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(MaxSharedMemoryPerMultiprocessor)");
  if ((e = cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
      cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(ReservedSharedMemoryPerBlock)");
  if ((e = cudaDeviceGetAttribute(&d.cooperative, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(CooperativeLaunch)");
  g_dev[dev] = d;
  *out = d;
  return QKNR_OK;
}

qknr_status configure_kernel(const void* fn, int dev, const DeviceInfo& di, int* regs) {
  std::lock_guard<std::mutex> lk(g_mu);
  const auto key = std::make_pair(fn, dev);
  auto it = g_configured.find(key);
  if (it == g_configured.end()) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)");
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
    it = g_configured.emplace(key, fa.numRegs).first;
  }
  *regs = it->second;
  return QKNR_OK;
}

qknr_status occupancy(const void* fn, int dev, int block, size_t smem, int* blocks_per_sm) {
  static std::map<std::tuple<const void*, int, int, size_t>, int> cache;
  const auto key = std::make_tuple(fn, dev, block, smem);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *blocks_per_sm = it->second;
      return QKNR_OK;
    }
  }
  int occ = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, block, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  std::lock_guard<std::mutex> lk(g_mu);
  cache[key] = occ;
  *blocks_per_sm = occ;
  return QKNR_OK;
}

qknr_status launch_kernel(const void* fn, int grid, int block, size_t smem, cudaStream_t stream, void** kargs,
                          bool overlap, const char* what) {
  // programmatic stream serialization: the kernel may launch while the
  // previous kernel in the stream finishes; it waits for that kernel
  // before its first global memory access (griddepcontrol.wait)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, kargs);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return QKNR_OK;
}

Span span_of(const void* base, long long rows, long long stride_bytes, long long row_bytes) {
  uintptr_t lo = reinterpret_cast<uintptr_t>(base);
  if (!base || rows <= 0 || row_bytes <= 0) return {lo, lo};
  return {lo, lo + static_cast<uintptr_t>((rows - 1) * stride_bytes + row_bytes)};
}

bool overlaps(Span a, Span b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

}  // namespace qknr_host

namespace {

using qknr_host::cuda_fail;
using qknr_host::DeviceInfo;
using qknr_host::fail;
using qknr_host::overlaps;
using qknr_host::Span;
using qknr_host::span_of;
using qknr_host::device_info;
using qknr_host::configure_kernel;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Plan {
  qknr::KernelParams kp;
  const void* fn = nullptr;
  int grid = 0, block = 0, smem = 0, stages = 0, ctas_per_sm = 0, warps = 0, group_warps = 0, regs = 0,
      num_sms = 0;
  bool launch = false;   // false: nothing to do
  char name[96];
};

qknr_status make_plan(const qknr_args* a, Plan* pl) {
  if (!a) return fail(QKNR_ERR_NULL, "args is NULL");
  if (a->abi_version != QKNR_ABI_VERSION)
    return fail(QKNR_ERR_ABI, "abi_version %u, library expects %d", a->abi_version, QKNR_ABI_VERSION);
  if (a->dtype != QKNR_BF16 && a->dtype != QKNR_FP16)
    return fail(QKNR_ERR_UNSUPPORTED, "activation dtype must be BF16 or FP16");
  if (a->cos_dtype != QKNR_FP32 && a->cos_dtype != QKNR_BF16)
    return fail(QKNR_ERR_UNSUPPORTED, "cos/sin dtype must be FP32 or BF16");
  if (a->cos_layout != QKNR_COS_SHARED_ROW && a->cos_layout != QKNR_COS_PER_HEAD_EXPANDED)
    return fail(QKNR_ERR_UNSUPPORTED, "unknown cos_layout %d", a->cos_layout);
  if (a->rope_style != QKNR_ROPE_INTERLEAVED && a->rope_style != QKNR_ROPE_ROTATE_HALF)
    return fail(QKNR_ERR_UNSUPPORTED, "unknown rope_style %d", a->rope_style);
  const int D = a->head_dim;
  if (D != 64 && D != 128) return fail(QKNR_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", D);
  if (a->tokens < 0) return fail(QKNR_ERR_SHAPE, "tokens < 0");
  if (a->n_heads_q < 0 || a->n_heads_k < 0 || a->n_heads_v < 0)
    return fail(QKNR_ERR_SHAPE, "negative head count");
  if (!(a->eps >= 0.0f)) return fail(QKNR_ERR_SHAPE, "eps must be >= 0");
  if (a->consumer_warps < 0 || a->consumer_warps > qknr::kMaxConsumerWarps)
    return fail(QKNR_ERR_SHAPE, "consumer_warps out of range 0..%d", qknr::kMaxConsumerWarps);
  if (a->stages < 0 || a->stages == 1 || a->stages > qknr::kMaxStages / 2)
    return fail(QKNR_ERR_SHAPE, "stages must be 0 (auto) or 2..%d", qknr::kMaxStages / 2);
  if (a->ctas_per_sm < 0 || a->ctas_per_sm > 4) return fail(QKNR_ERR_SHAPE, "ctas_per_sm out of range 0..4");
  if (a->group_warps < 0 || a->group_warps > qknr::kMaxConsumerWarps ||
      (a->group_warps && a->consumer_warps && a->consumer_warps % a->group_warps))
    return fail(QKNR_ERR_SHAPE, "group_warps must divide consumer_warps");

  const int es = 2;
  const int ces = a->cos_dtype == QKNR_FP32 ? 4 : 2;
  const long long T = a->tokens;
  const int hq = a->n_heads_q, hk = a->n_heads_k;
  const bool expanded = a->cos_layout == QKNR_COS_PER_HEAD_EXPANDED;

  const bool rh = a->rope_style == QKNR_ROPE_ROTATE_HALF;
  const bool bf16_tab = a->cos_dtype == QKNR_BF16;
  if (a->dtype == QKNR_BF16)
    pl->fn = bf16_tab ? qknr::kernel_bf16_bf16(D, rh, expanded) : qknr::kernel_bf16_f32(D, rh, expanded);
  else
    pl->fn = bf16_tab ? qknr::kernel_fp16_bf16(D, rh, expanded) : qknr::kernel_fp16_f32(D, rh, expanded);
  if (!pl->fn) return fail(QKNR_ERR_UNSUPPORTED, "no kernel instance for this combination");
  snprintf(pl->name, sizeof(pl->name), "qknr_fused<%s,%s,D%d,%s,%s>", a->dtype == QKNR_BF16 ? "bf16" : "fp16",
           bf16_tab ? "bf16" : "fp32", D, rh ? "rotate_half" : "interleaved", expanded ? "expanded" : "shared");
  memset(&pl->kp, 0, sizeof(pl->kp));
  pl->launch = false;
  if (T == 0) return QKNR_OK;   // nothing to read or write: pointers may be NULL

  // outputs default to in place
  const void* q = a->q;
  const void* k = a->k;
  const void* v = a->v;
  void* q_out = a->q_out ? a->q_out : const_cast<void*>(q);
  void* k_out = a->k_out ? a->k_out : const_cast<void*>(k);
  const long long qs = a->q_stride ? a->q_stride : (long long)hq * D;
  const long long ks = a->k_stride ? a->k_stride : (long long)hk * D;
  const long long vs = a->v_stride ? a->v_stride : (long long)a->n_heads_v * D;
  const long long qos = a->q_out_stride ? a->q_out_stride : qs;
  const long long kos = a->k_out_stride ? a->k_out_stride : ks;
  const long long vos = a->v_out_stride ? a->v_out_stride : vs;
  const bool copy_v = a->n_heads_v > 0 && a->v_out && !(a->v_out == v && vos == vs);
  const int hv = copy_v ? a->n_heads_v : 0;

  if (hq > 0 && (!q || !a->gamma_q)) return fail(QKNR_ERR_NULL, "q and gamma_q are required when n_heads_q > 0");
  if (hk > 0 && (!k || !a->gamma_k)) return fail(QKNR_ERR_NULL, "k and gamma_k are required when n_heads_k > 0");
  if (copy_v && !v) return fail(QKNR_ERR_NULL, "v is required to copy V into v_out");
  if (hq + hk > 0 && (!a->cos || !a->sin)) return fail(QKNR_ERR_NULL, "cos and sin are required");
  if (hq > 0 && qs < (long long)hq * D) return fail(QKNR_ERR_SHAPE, "q_stride < n_heads_q * head_dim");
  if (hk > 0 && ks < (long long)hk * D) return fail(QKNR_ERR_SHAPE, "k_stride < n_heads_k * head_dim");
  if (hq > 0 && qos < (long long)hq * D) return fail(QKNR_ERR_SHAPE, "q_out_stride too small");
  if (hk > 0 && kos < (long long)hk * D) return fail(QKNR_ERR_SHAPE, "k_out_stride too small");
  if (hv > 0 && (vs < (long long)hv * D || vos < (long long)hv * D))
    return fail(QKNR_ERR_SHAPE, "v strides too small");
  if (expanded && hq > 0 && hk > 0 && hq != hk)
    return fail(QKNR_ERR_SHAPE, "per-head expanded tables need n_heads_q == n_heads_k");
  const long long cos_rows = a->cos_rows ? a->cos_rows : T;
  if (a->cos_rows < 0) return fail(QKNR_ERR_SHAPE, "cos_rows < 0");

  // alignment: every bulk copy and 16-byte store starts on a 16-byte boundary
  if (hq > 0 && (!aligned16(q) || !aligned16(q_out) || (qs * es) % 16 || (qos * es) % 16))
    return fail(QKNR_ERR_ALIGN, "q / q_out base or row stride not 16-byte aligned");
  if (hk > 0 && (!aligned16(k) || !aligned16(k_out) || (ks * es) % 16 || (kos * es) % 16))
    return fail(QKNR_ERR_ALIGN, "k / k_out base or row stride not 16-byte aligned");
  if (hv > 0 && (!aligned16(v) || !aligned16(a->v_out) || (vs * es) % 16 || (vos * es) % 16))
    return fail(QKNR_ERR_ALIGN, "v / v_out base or row stride not 16-byte aligned");
  if (hq + hk > 0 && (!aligned16(a->cos) || !aligned16(a->sin)))
    return fail(QKNR_ERR_ALIGN, "cos / sin not 16-byte aligned");
  if ((a->gamma_q && (reinterpret_cast<uintptr_t>(a->gamma_q) & 3u)) ||
      (a->gamma_k && (reinterpret_cast<uintptr_t>(a->gamma_k) & 3u)))
    return fail(QKNR_ERR_ALIGN, "gamma not 4-byte aligned");

  pl->launch = T > 0 && (hq + hk + hv) > 0;
  const int table_heads = expanded ? (hq > hk ? hq : hk) : 1;
  const long long cos_row_bytes = hq + hk > 0 ? (long long)table_heads * D * ces : 0;

  // overlap: an output that is not exactly its own input must not touch any input
  if (pl->launch) {
    const Span in[] = {
        span_of(q, hq ? T : 0, qs * es, (long long)hq * D * es),
        span_of(k, hk ? T : 0, ks * es, (long long)hk * D * es),
        span_of(v, hv ? T : 0, vs * es, (long long)hv * D * es),
        span_of(a->cos, hq + hk ? cos_rows : 0, cos_row_bytes, cos_row_bytes),
        span_of(a->sin, hq + hk ? cos_rows : 0, cos_row_bytes, cos_row_bytes),
        span_of(a->gamma_q, hq ? 1 : 0, 0, (long long)D * 4),
        span_of(a->gamma_k, hk ? 1 : 0, 0, (long long)D * 4),
    };
    struct {
      const void* out;
      const void* own;
      long long os, is, heads;
      const char* name;
    } outs[] = {{q_out, q, qos, qs, hq, "q_out"}, {k_out, k, kos, ks, hk, "k_out"},
                {a->v_out, v, vos, vs, hv, "v_out"}};
    for (auto& o : outs) {
      if (o.heads == 0) continue;
      if (o.out == o.own && o.os == o.is) continue;   // exactly in place
      const Span so = span_of(o.out, T, o.os * es, o.heads * D * es);
      for (const Span& si : in)
        if (overlaps(so, si)) return fail(QKNR_ERR_OVERLAP, "%s overlaps an input without being in place", o.name);
    }
  }

  // stage layout
  const unsigned q_bytes = hq * D * es, k_bytes = hk * D * es, v_bytes = hv * D * es;
  const long long tx = (long long)q_bytes + k_bytes + v_bytes + 2 * cos_row_bytes;
  const long long stage_bytes = (tx + qknr::kStageAlign - 1) / qknr::kStageAlign * qknr::kStageAlign;

  qknr::KernelParams& kp = pl->kp;
  kp.q = static_cast<const char*>(q);
  kp.k = static_cast<const char*>(k);
  kp.v = static_cast<const char*>(v);
  kp.q_out = static_cast<char*>(q_out);
  kp.k_out = static_cast<char*>(k_out);
  kp.v_out = static_cast<char*>(a->v_out);
  kp.q_stride = qs * es;
  kp.k_stride = ks * es;
  kp.v_stride = vs * es;
  kp.q_out_stride = qos * es;
  kp.k_out_stride = kos * es;
  kp.v_out_stride = vos * es;
  kp.tokens = T;
  kp.cos_rows = cos_rows > 0 ? cos_rows : 1;
  kp.cos = static_cast<const char*>(a->cos);
  kp.sin = static_cast<const char*>(a->sin);
  kp.cos_row_bytes = cos_row_bytes;
  kp.gamma_q = a->gamma_q;
  kp.gamma_k = a->gamma_k;
  kp.status = a->dev_status;
  kp.wait_limit_ns = a->wait_limit_ns ? a->wait_limit_ns : 2000000000ull;
  kp.eps = a->eps;
  kp.inv_d = 1.0f / static_cast<float>(D);
  kp.hq = hq;
  kp.hk = hk;
  kp.hv = hv;
  kp.flags = a->flags;
  kp.qk_merged = hq > 0 && hk > 0 && static_cast<const char*>(k) == static_cast<const char*>(q) + q_bytes &&
                 ks == qs;
  kp.off_k = q_bytes;
  kp.off_v = q_bytes + k_bytes;
  kp.off_cos = q_bytes + k_bytes + v_bytes;
  kp.off_sin = kp.off_cos + static_cast<unsigned>(cos_row_bytes);
  kp.stage_bytes = static_cast<unsigned>(stage_bytes);
  // buffer spans for checked builds
  auto ms = [](Span x) { return qknr::MemSpan{x.lo, x.hi}; };
  kp.sp_q = ms(span_of(q, hq ? T : 0, qs * es, (long long)hq * D * es));
  kp.sp_k = ms(span_of(k, hk ? T : 0, ks * es, (long long)hk * D * es));
  kp.sp_v = ms(span_of(v, hv ? T : 0, vs * es, (long long)hv * D * es));
  kp.sp_q_out = ms(span_of(q_out, hq ? T : 0, qos * es, (long long)hq * D * es));
  kp.sp_k_out = ms(span_of(k_out, hk ? T : 0, kos * es, (long long)hk * D * es));
  kp.sp_v_out = ms(span_of(a->v_out, hv ? T : 0, vos * es, (long long)hv * D * es));
  kp.sp_cos = ms(span_of(a->cos, hq + hk ? cos_rows : 0, cos_row_bytes, cos_row_bytes));
  kp.sp_sin = ms(span_of(a->sin, hq + hk ? cos_rows : 0, cos_row_bytes, cos_row_bytes));
  kp.sp_gq = ms(span_of(a->gamma_q, hq ? 1 : 0, 0, (long long)D * 4));
  kp.sp_gk = ms(span_of(a->gamma_k, hk ? 1 : 0, 0, (long long)D * 4));
  if ((a->flags & QKNR_FLAG_TEST_SHORT_OUT) && T > 1)
    kp.sp_q_out = ms(span_of(q_out, hq ? T - 1 : 0, qos * es, (long long)hq * D * es));
  kp.tx_bytes = static_cast<unsigned>(tx);

  return QKNR_OK;
}

// Device-dependent part of the plan: grid, ring depth and shared memory.
qknr_status size_launch(const qknr_args* a, Plan* pl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceInfo di;
  qknr_status st = device_info(dev, &di);
  if (st != QKNR_OK) return st;
  st = configure_kernel(pl->fn, dev, di, &pl->regs);
  if (st != QKNR_OK) return st;
  pl->num_sms = di.num_sms;

  // Defaults from sweeps on GB300.  Rows of many heads (>= 32 passes of
  // heads per row, e.g. Wan's 40 Q + 40 K heads of 128) run best with all
  // 12 consumer warps on one row and a 4-deep ring: DRAM is the limit and
  // more bytes in flight only queue.  Rows of few heads leave each warp too
  // little work per row, so 16 warps form groups of about 6 passes per
  // warp that each take whole rows, several rows in flight.  One CTA per SM
  // (a second does not fit beside the first one's registers).
  const int hpw = 32 / (a->head_dim / 8);
  const int nq = (pl->kp.hq + hpw - 1) / hpw, nk = (pl->kp.hk + hpw - 1) / hpw;
  const int passes = nq + nk;
  const bool wide_rows = passes >= 32 || passes == 0;
  const int warps = a->consumer_warps ? a->consumer_warps : (wide_rows ? 12 : 16);
  const long long rows_per_cta_1 = (a->tokens + di.num_sms - 1) / di.num_sms;   // at one CTA per SM
  const int cps = a->ctas_per_sm ? a->ctas_per_sm : 1;
  const long long stage_bytes = pl->kp.stage_bytes;
  // shared memory one CTA may use when `cps` CTAs share an SM
  long long budget = di.smem_per_sm / cps - di.smem_reserved;
  if (budget > di.smem_optin) budget = di.smem_optin;
  const long long ring = budget - qknr::kOffStage0;
  const long long fit = ring > 0 ? ring / stage_bytes : 0;
  const long long grid0 = (long long)di.num_sms * cps;
  const long long rows_per_cta = (a->tokens + grid0 - 1) / grid0;

  // Wide rows that carry a V copy, a per-head expanded table, or that a CTA
  // sees few of, do better as two groups of two stages (sweeps: Wan out of
  // place 329 vs 350 us, Wan with a bf16 expanded table 326 vs 343 us,
  // FLUX.2 Q+K in one launch 73.8 vs 76.1 us) where two such rings fit (an
  // fp32 expanded table's stages do not: one group of three); a deeper ring
  // than four stages in all only queues more reads (Wan 231 vs 211 us with
  // six).
  const bool expanded = a->cos_layout == QKNR_COS_PER_HEAD_EXPANDED;
  const bool two_groups = wide_rows && passes > 0 && (pl->kp.hv > 0 || expanded || rows_per_cta_1 < 128);
  // rows with a V copy that a CTA sees many of: three groups of two stages
  // (Wan out of place 321 vs 329 us; with few rows per CTA, FLUX.2, two)
  const bool three_groups = two_groups && pl->kp.hv > 0 && rows_per_cta_1 >= 128;
  int gw = a->group_warps;
  if (gw == 0) {
    int want = three_groups ? warps / 3
               : two_groups ? warps / 2
                            : (wide_rows ? warps : (passes + 5) / 6);   // narrow: ~6 passes per warp
    if (want < 1) want = 1;
    gw = warps;
    for (int g = want; g <= warps; ++g)
      if (warps % g == 0) {
        gw = g;
        break;
      }
    // every group needs a ring of at least two stages, and no more groups
    // than the rows a CTA will see
    while (gw < warps && (2LL * (warps / gw) > fit || 2 * (warps / gw) > qknr::kMaxStages ||
                          warps / gw > rows_per_cta)) {
      int g = gw + 1;
      while (warps % g) ++g;
      gw = g;
    }
  }
  if (warps % gw) return fail(QKNR_ERR_SHAPE, "group_warps %d does not divide consumer_warps %d", gw, warps);
  const int n_groups = warps / gw;

  // ring depth per group: four stages in all for wide rows (one group of 4
  // or two of 2), else about 128 KB of stages in all; at least two each
  int stages = a->stages;
  if (stages == 0) {
    long long want = wide_rows ? 4 / n_groups : (128 * 1024) / (stage_bytes * n_groups);
    if (want < 2) want = 2;
    if (want > 8) want = 8;
    long long cap = fit / n_groups;
    if (cap > qknr::kMaxStages / n_groups) cap = qknr::kMaxStages / n_groups;
    stages = static_cast<int>(cap < want ? cap : want);
    // no deeper than the rows one group will see
    const long long rows_per_group = (rows_per_cta + n_groups - 1) / n_groups;
    if (rows_per_group >= 2 && stages > rows_per_group) stages = static_cast<int>(rows_per_group);
    if (stages < 2) stages = 2;
  }
  if (stages * n_groups > qknr::kMaxStages)
    return fail(QKNR_ERR_SHAPE, "%d groups x %d stages exceeds %d stages", n_groups, stages, qknr::kMaxStages);
  const long long smem = qknr::kOffStage0 + static_cast<long long>(stages) * n_groups * stage_bytes;
  if (smem > di.smem_optin)
    return fail(QKNR_ERR_UNSUPPORTED,
                "%d groups x %d stages of %lld-byte rows need %lld B of shared memory (max %d)", n_groups, stages,
                stage_bytes, smem, di.smem_optin);
  const int block = 32 * (warps + 1);
  int occ = 0;
  st = qknr_host::occupancy(pl->fn, dev, block, static_cast<size_t>(smem), &occ);
  if (st != QKNR_OK) return st;
  if (occ < 1) return fail(QKNR_ERR_UNSUPPORTED, "kernel does not fit on an SM with %lld B shared memory", smem);
  const int per_sm = cps < occ ? cps : occ;
  long long grid = (long long)di.num_sms * per_sm;
  if (grid > a->tokens) grid = a->tokens;
  pl->kp.stages = stages;
  pl->kp.consumer_warps = warps;
  pl->kp.group_warps = gw;
  // Before its dependency wait a CTA asks L2 for its second ring fill (rows
  // ring .. 2 ring - 1 of its own), when it has at least four fills of rows.
  // Under programmatic dependent launch that read overlaps the previous
  // kernel's last rows: back to back, Wan 208.3 -> 207.5 us, the FLUX.2
  // per-tensor pair 75.7 -> 71.2 us, Q and K in one launch 71.8 -> 69.2 us.
  // Prefetching the first fill instead (which the producer's own copies
  // request right after the wait) gained less on the pair (73.2 us), and
  // shorter launches, whose inputs the previous kernel often leaves in L2,
  // only lose (4096 x 24 x 128 back to back 14.1 -> 15.2 us).  A call that
  // starts cold (after an L2 flush, nothing to overlap) loses about 1 us:
  // Wan 8192 x 40 x 128 60.8 -> 62.0 us, the FLUX.2 Q launch 43.3 -> 43.8.
  const long long ring_rows = static_cast<long long>(stages) * n_groups;
  const long long cta_rows = (a->tokens + grid - 1) / grid;
  pl->kp.prefetch_rows =
      !(a->flags & QKNR_FLAG_NO_PREFETCH) && cta_rows >= 4 * ring_rows ? static_cast<int>(ring_rows) : 0;
  // split a group's warps between Q and K in proportion to their passes
  if (nq == 0 || nk == 0) {
    pl->kp.warps_q = nq ? gw : 0;
    pl->kp.warps_k = nk ? gw : 0;
  } else if (gw == 1) {
    pl->kp.warps_q = pl->kp.warps_k = 1;
  } else {
    int wq = static_cast<int>((static_cast<long long>(gw) * nq + (nq + nk) / 2) / (nq + nk));
    wq = wq < 1 ? 1 : (wq > gw - 1 ? gw - 1 : wq);
    pl->kp.warps_q = wq;
    pl->kp.warps_k = gw - wq;
  }
  pl->grid = static_cast<int>(grid);
  pl->block = block;
  pl->smem = static_cast<int>(smem);
  pl->kp.smem_bytes = static_cast<unsigned>(smem);
  pl->stages = stages;
  pl->ctas_per_sm = per_sm;
  pl->warps = warps;
  pl->group_warps = gw;
  return QKNR_OK;
}

}  // namespace

extern "C" {

void qknr_args_init(qknr_args* a) {
  if (!a) return;
  memset(a, 0, sizeof(*a));
  a->abi_version = QKNR_ABI_VERSION;
  a->dtype = QKNR_BF16;
  a->eps = 1e-6f;
  a->cos_dtype = QKNR_FP32;
  a->cos_layout = QKNR_COS_SHARED_ROW;
  a->rope_style = QKNR_ROPE_INTERLEAVED;
}

qknr_status qknr_query(const qknr_args* args, qknr_launch_info* info) {
  if (!info) return fail(QKNR_ERR_NULL, "info is NULL");
  memset(info, 0, sizeof(*info));
  Plan pl;
  qknr_status st = make_plan(args, &pl);
  if (st != QKNR_OK) return st;
  snprintf(info->kernel, sizeof(info->kernel), "%s", pl.name);
  info->stage_bytes = static_cast<int32_t>(pl.kp.stage_bytes);
  if (!pl.launch) return QKNR_OK;
  st = size_launch(args, &pl);
  if (st != QKNR_OK) return st;
  info->grid = pl.grid;
  info->block = pl.block;
  info->dyn_smem = pl.smem;
  info->stages = pl.stages;
  info->ctas_per_sm = pl.ctas_per_sm;
  info->consumer_warps = pl.warps;
  info->group_warps = pl.group_warps;
  info->registers = pl.regs;
  info->num_sms = pl.num_sms;
  info->prefetch_rows = pl.kp.prefetch_rows;
  return QKNR_OK;
}

qknr_status qknr_forward(const qknr_args* args, qknr_stream_t stream) {
  Plan pl;
  qknr_status st = make_plan(args, &pl);
  if (st != QKNR_OK || !pl.launch) return st;
  st = size_launch(args, &pl);
  if (st != QKNR_OK) return st;
  void* kargs[] = {&pl.kp};
  return qknr_host::launch_kernel(pl.fn, pl.grid, pl.block, static_cast<size_t>(pl.smem),
                                  reinterpret_cast<cudaStream_t>(stream), kargs,
                                  !(args->flags & qknr::kFlagNoOverlap), "cudaLaunchKernelExC");
}

const char* qknr_status_string(int32_t s) {
  switch (s) {
    case QKNR_OK: return "ok";
    case QKNR_ERR_NULL: return "required pointer is NULL";
    case QKNR_ERR_SHAPE: return "size, count or stride out of range";
    case QKNR_ERR_ALIGN: return "address or row stride not 16-byte aligned";
    case QKNR_ERR_UNSUPPORTED: return "unsupported combination";
    case QKNR_ERR_CUDA: return "CUDA runtime error";
    case QKNR_ERR_TIMEOUT: return "in-kernel wait timed out";
    case QKNR_ERR_OVERLAP: return "output overlaps an input";
    case QKNR_ERR_ABI: return "ABI version mismatch";
    case QKNR_ERR_BOUNDS: return "access outside a buffer (checked build)";
    default: return "unknown status";
  }
}

const char* qknr_last_error(void) { return qknr_host::g_err; }

int32_t qknr_abi_version(void) { return QKNR_ABI_VERSION; }

size_t qknr_sizeof_args(void) { return sizeof(qknr_args); }

size_t qknr_sizeof_launch_info(void) { return sizeof(qknr_launch_info); }

}  // extern "C"
