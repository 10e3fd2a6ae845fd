// C-ABI launcher of the AdaLN scale/shift kernel: validation, launch
// planning and the launch.  No allocation, no synchronisation.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>

#include "../../include/qknr_adaln.h"
#include "adaln_kernel.cuh"
#include "qknr_host.h"

namespace qknr {
const void* adaln_kernel_for(int act, bool mod_fp32, int cpl);
}

namespace {

using qknr_host::aligned16;
using qknr_host::fail;
using qknr_host::Span;
using qknr_host::span_of;

struct AdaPlan {
  qknr::AdaLNParams kp;
  const void* fn = nullptr;
  int grid = 0, block = 0, smem = 0, stages = 0, ctas_per_sm = 0, warps = 0, group_warps = 0, regs = 0,
      num_sms = 0, stage_bytes = 0, cpl = 0;
  bool launch = false;
};

qknr_status plan(const qknr_adaln_args* a, AdaPlan* pl, bool size_device) {
  if (!a) return fail(QKNR_ERR_NULL, "args is NULL");
  if (a->abi_version != QKNR_ABI_VERSION)
    return fail(QKNR_ERR_ABI, "abi_version %u, library expects %d", a->abi_version, QKNR_ABI_VERSION);
  if (a->dtype != QKNR_BF16 && a->dtype != QKNR_FP16)
    return fail(QKNR_ERR_UNSUPPORTED, "activation dtype must be BF16 or FP16");
  if (a->mod_dtype != QKNR_FP32 && a->mod_dtype != a->dtype)
    return fail(QKNR_ERR_UNSUPPORTED, "scale/shift dtype must be FP32 or the activation dtype");
  const int C = a->hidden;
  if (C < 8 || C % 8 || C > 32768) return fail(QKNR_ERR_UNSUPPORTED, "hidden %d (a multiple of 8, <= 32768)", C);
  if (a->tokens < 0 || a->rows_per_batch < 0) return fail(QKNR_ERR_SHAPE, "negative tokens or rows_per_batch");
  if (!(a->eps >= 0.0f)) return fail(QKNR_ERR_SHAPE, "eps must be >= 0");
  if (a->consumer_warps < 0 || a->consumer_warps > qknr::kAdaMaxWarps)
    return fail(QKNR_ERR_SHAPE, "consumer_warps out of range 0..%d", qknr::kAdaMaxWarps);
  if (a->group_warps < 0 || a->group_warps > qknr::kAdaMaxWarps ||
      (a->group_warps && a->consumer_warps && a->consumer_warps % a->group_warps))
    return fail(QKNR_ERR_SHAPE, "group_warps must divide consumer_warps");
  if (a->stages < 0 || a->stages == 1 || a->stages > qknr::kAdaMaxStages / 2)
    return fail(QKNR_ERR_SHAPE, "stages must be 0 (auto) or 2..%d", qknr::kAdaMaxStages / 2);
  if (a->ctas_per_sm < 0 || a->ctas_per_sm > 4) return fail(QKNR_ERR_SHAPE, "ctas_per_sm out of range 0..4");
  memset(&pl->kp, 0, sizeof(pl->kp));
  pl->launch = false;
  const long long T = a->tokens;
  if (T == 0) return QKNR_OK;

  const int es = 2, mes = a->mod_dtype == QKNR_FP32 ? 4 : 2;
  const void* out = a->out ? a->out : a->x;
  const long long xs = a->x_stride ? a->x_stride : C;
  const long long os = a->out_stride ? a->out_stride : xs;
  const long long ms = a->mod_stride ? a->mod_stride : C;
  const long long rpb = a->rows_per_batch ? a->rows_per_batch : T;
  const long long B = (T + rpb - 1) / rpb;
  if (!a->x || !a->scale || !a->shift) return fail(QKNR_ERR_NULL, "x, scale and shift are required");
  if (xs < C || os < C || ms < C) return fail(QKNR_ERR_SHAPE, "a stride is smaller than hidden");
  if (!aligned16(a->x) || !aligned16(out) || !aligned16(a->scale) || !aligned16(a->shift) || (xs * es) % 16 ||
      (os * es) % 16 || (ms * mes) % 16)
    return fail(QKNR_ERR_ALIGN, "x / out / scale / shift base or stride not 16-byte aligned");
  const bool in_place = out == a->x && os == xs;
  if (!in_place) {
    const Span so = span_of(out, T, os * es, (long long)C * es);
    const Span in[] = {span_of(a->x, T, xs * es, (long long)C * es), span_of(a->scale, B, ms * mes, (long long)C * mes),
                       span_of(a->shift, B, ms * mes, (long long)C * mes)};
    for (const Span& si : in)
      if (qknr_host::overlaps(so, si)) return fail(QKNR_ERR_OVERLAP, "out overlaps an input without being in place");
  }

  qknr::AdaLNParams& kp = pl->kp;
  kp.x = static_cast<const char*>(a->x);
  kp.out = static_cast<char*>(const_cast<void*>(out));
  kp.x_stride = xs * es;
  kp.out_stride = os * es;
  kp.tokens = T;
  kp.rows_per_batch = rpb;
  kp.scale = static_cast<const char*>(a->scale);
  kp.shift = static_cast<const char*>(a->shift);
  kp.mod_stride = ms * mes;
  kp.status = a->dev_status;
  kp.wait_limit_ns = a->wait_limit_ns ? a->wait_limit_ns : 2000000000ull;
  kp.eps = a->eps;
  kp.inv_c = 1.0f / static_cast<float>(C);
  kp.hidden = C;
  kp.flags = a->flags;
  kp.row_bytes = static_cast<unsigned>(C * es);
  kp.stage_bytes = (kp.row_bytes + qknr::kAdaStageAlign - 1) / qknr::kAdaStageAlign * qknr::kAdaStageAlign;
  // buffer spans for checked builds
  auto msp = [](Span x) { return qknr::MemSpan{x.lo, x.hi}; };
  kp.sp_x = msp(span_of(a->x, T, xs * es, (long long)C * es));
  kp.sp_out = msp(span_of(out, T, os * es, (long long)C * es));
  kp.sp_scale = msp(span_of(a->scale, B, ms * mes, (long long)C * mes));
  kp.sp_shift = msp(span_of(a->shift, B, ms * mes, (long long)C * mes));
  pl->stage_bytes = static_cast<int>(kp.stage_bytes);
  pl->launch = true;
  if (!size_device) return QKNR_OK;

  // ---- device-dependent sizing
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return qknr_host::cuda_fail(e, "cudaGetDevice");
  qknr_host::DeviceInfo di;
  qknr_status st = qknr_host::device_info(dev, &di);
  if (st != QKNR_OK) return st;
  pl->num_sms = di.num_sms;
  const int n_chunks = C / 8;
  // Default (sweeps on GB300, hidden 5120 and 6144): one CTA per SM of 16
  // consumer warps in groups of about 12 chunks per lane (2 warps), 2 stages
  // each.  The producer hands each row to whichever group has a free stage,
  // which balances the groups of a CTA; two CTAs of 8 warps per SM, the
  // earlier default, end far apart (the second CTA on an SM gets the smaller
  // share of it): 47.5 vs 45.7 us on FLUX.2, 117.3 vs 115.5 us on Wan.
  int warps = a->consumer_warps, cps = a->ctas_per_sm;
  if (!warps) warps = 16;
  if (!cps) cps = 1;
  long long budget = di.smem_per_sm / cps - di.smem_reserved;
  if (budget > di.smem_optin) budget = di.smem_optin;
  const long long fit = (budget - qknr::kAdaOffStage0) / kp.stage_bytes;
  const long long grid0 = (long long)di.num_sms * cps;
  const long long rows_per_cta = (T + grid0 - 1) / grid0;
  // Group size (sweeps on GB300, hidden 5120 and 6144): about 12 chunks of
  // 16 bytes per lane, i.e. 2 warps per row and 8 rows in flight with 16
  // warps; at most 8 groups, two stages each that fit, and no more groups
  // than the rows a CTA sees.
  int gw = a->group_warps;
  if (gw == 0) {
    const int want = (n_chunks + 32 * 12 - 1) / (32 * 12);
    gw = warps;
    for (int g = want < 1 ? 1 : want; g <= warps; ++g) {
      if (warps % g) continue;
      const int ng = warps / g;
      if (ng <= qknr::kAdaMaxGroups && 2LL * ng <= fit && ng <= rows_per_cta) {
        gw = g;
        break;
      }
    }
  }
  if (warps % gw) return fail(QKNR_ERR_SHAPE, "group_warps %d does not divide consumer_warps %d", gw, warps);
  const int n_groups = warps / gw;
  if (n_groups > qknr::kAdaMaxGroups) return fail(QKNR_ERR_SHAPE, "more than %d row groups", qknr::kAdaMaxGroups);
  const int cpl = (n_chunks + 32 * gw - 1) / (32 * gw);
  // ring depth per group: up to 4, at least 2
  int stages = a->stages;
  if (stages == 0) {
    long long cap = fit / n_groups;
    if (cap > qknr::kAdaMaxStages / n_groups) cap = qknr::kAdaMaxStages / n_groups;
    stages = static_cast<int>(cap < 4 ? cap : 4);
    const long long rows_per_group = (rows_per_cta + n_groups - 1) / n_groups;
    if (rows_per_group >= 2 && stages > rows_per_group) stages = static_cast<int>(rows_per_group);
    if (stages < 2) stages = 2;
  }
  if (stages * n_groups > qknr::kAdaMaxStages)
    return fail(QKNR_ERR_SHAPE, "%d groups x %d stages exceeds %d stages", n_groups, stages, qknr::kAdaMaxStages);
  const long long smem = qknr::kAdaOffStage0 + static_cast<long long>(stages) * n_groups * kp.stage_bytes;
  if (smem > di.smem_optin)
    return fail(QKNR_ERR_UNSUPPORTED, "%d groups x %d stages of %u-byte rows need %lld B of shared memory (max %d)",
                n_groups, stages, kp.stage_bytes, smem, di.smem_optin);
  const int unroll = cpl >= 4 ? 4 : (cpl >= 2 ? 2 : 1);
  pl->fn = qknr::adaln_kernel_for(a->dtype == QKNR_BF16 ? 0 : 1, a->mod_dtype == QKNR_FP32, unroll);
  if (!pl->fn) return fail(QKNR_ERR_UNSUPPORTED, "no kernel instance for this combination");
  st = qknr_host::configure_kernel(pl->fn, dev, di, &pl->regs);
  if (st != QKNR_OK) return st;
  const int block = 32 * (warps + 1);
  int occ = 0;
  st = qknr_host::occupancy(pl->fn, dev, block, static_cast<size_t>(smem), &occ);
  if (st != QKNR_OK) return st;
  if (occ < 1) return fail(QKNR_ERR_UNSUPPORTED, "kernel does not fit on an SM with %lld B shared memory", smem);
  const int per_sm = cps < occ ? cps : occ;
  long long grid = (long long)di.num_sms * per_sm;
  if (grid > T) grid = T;
  kp.consumer_warps = warps;
  kp.group_warps = gw;
  kp.stages = stages;
  // Before its dependency wait each CTA asks L2 for its first four rows of
  // x (sweeps on GB300 against none: Wan 107.0 -> 106.6 us back to back,
  // FLUX.2 45.2 -> 44.9 us flushed and 39.9 -> 38.7 us back to back; two,
  // six or eight rows about the same, the whole first ring fill of 16 rows
  // or the second fill slower on Wan and flushed)
  const bool no_prefetch = (a->flags & (QKNR_FLAG_NO_OVERLAP | QKNR_FLAG_NO_PREFETCH)) != 0;
  kp.prefetch_rows = no_prefetch ? 0 : 4;
  pl->grid = static_cast<int>(grid);
  pl->block = block;
  pl->smem = static_cast<int>(smem);
  kp.smem_bytes = static_cast<unsigned>(smem);
  pl->stages = stages;
  pl->ctas_per_sm = per_sm;
  pl->warps = warps;
  pl->group_warps = gw;
  pl->cpl = cpl;
  return QKNR_OK;
}

}  // namespace

extern "C" {

void qknr_adaln_args_init(qknr_adaln_args* a) {
  if (!a) return;
  memset(a, 0, sizeof(*a));
  a->abi_version = QKNR_ABI_VERSION;
  a->dtype = QKNR_BF16;
  a->mod_dtype = QKNR_BF16;
  a->eps = 1e-6f;
}

qknr_status qknr_adaln_query(const qknr_adaln_args* args, qknr_launch_info* info) {
  if (!info) return fail(QKNR_ERR_NULL, "info is NULL");
  memset(info, 0, sizeof(*info));
  AdaPlan pl;
  qknr_status st = plan(args, &pl, false);
  if (st != QKNR_OK) return st;
  info->stage_bytes = pl.stage_bytes;
  if (!pl.launch) return QKNR_OK;
  st = plan(args, &pl, true);
  if (st != QKNR_OK) return st;
  snprintf(info->kernel, sizeof(info->kernel), "adaln<%s,%s,cpl%d>", args->dtype == QKNR_BF16 ? "bf16" : "fp16",
           args->mod_dtype == QKNR_FP32 ? "fp32" : "act", pl.cpl);
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

qknr_status qknr_adaln_forward(const qknr_adaln_args* args, qknr_stream_t stream) {
  AdaPlan pl;
  qknr_status st = plan(args, &pl, false);
  if (st != QKNR_OK || !pl.launch) return st;
  st = plan(args, &pl, true);
  if (st != QKNR_OK) return st;
  void* kargs[] = {&pl.kp};
  return qknr_host::launch_kernel(pl.fn, pl.grid, pl.block, static_cast<size_t>(pl.smem),
                                  reinterpret_cast<cudaStream_t>(stream), kargs, !(args->flags & QKNR_FLAG_NO_OVERLAP),
                                  "cudaLaunchKernelExC(AdaLN)");
}

size_t qknr_adaln_sizeof_args(void) { return sizeof(qknr_adaln_args); }

}  // extern "C"
