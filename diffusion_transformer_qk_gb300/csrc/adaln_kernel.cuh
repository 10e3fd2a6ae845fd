// AdaLN scale/shift kernel for sm_103a: per token row, a layer norm without
// affine over the hidden dimension followed by the per-sample modulation
//
//     out[c] = (x[c] - mean) * rsqrt(var + eps) * (1 + scale[b, c]) + shift[b, c]
//
// ("fused qknorm rope Flux 2.0", section "Not in this PR — follow-ups":
// AdaLN's fuse_scale_shift, 81 calls per FLUX.2 step).
//
// Same streaming structure as the QK kernel: a persistent CTA per SM, one
// producer lane bulk-copying token rows into per-group shared-memory rings,
// consumer warps in groups that each take whole rows, so several rows are
// in flight.  The producer gives each of the CTA's rows (blockIdx.x,
// blockIdx.x + gridDim.x, ...) to whichever group has a free stage first,
// writing the row's index beside the stage; a group that works faster
// takes more rows, and when the rows run out each group's next stage
// carries an end mark.  Lane l of warp w of a group of GW warps handles the 16-byte
// chunks k = (w*32 + l) + i*32*GW of the staged row.
//
// Statistics in one pass over the staged row (moments.cuh): each thread
// sums x - k and (x - k)^2 over its values around its own first value k,
// which gives its count, its mean relative to the row's shift K (the lower
// median of its first 8 values) and its sum of squared deviations; these parts are merged by shuffles
// inside a warp and, through shared memory and one named barrier, across
// the group's warps, into m1 = mean - K and var.  A second pass over
// the staged row writes ((x - K) * r - m1 * r) * (1 + scale) + shift with
// r = rsqrt(var + eps), and the stage goes back to the producer after that
// pass.
//
// Every mbarrier wait is bounded.  The decision to continue is collective:
// each warp posts whether its wait succeeded with its partial sums, and
// the group leaves the row loop together when any warp failed, so no warp
// can be left waiting at a named barrier for one that gave up.
#pragma once

#include "moments.cuh"
#include "qknr_ptx.cuh"
#include "rings.cuh"

namespace qknr {

constexpr int kAdaMaxWarps = 16;
constexpr int kAdaMaxThreads = 32 * (kAdaMaxWarps + 1);
constexpr int kAdaMaxStages = 32;                 // all groups' rings together
constexpr int kAdaMaxGroups = 8;                  // named barriers 1..8
// dynamic shared memory map (bytes)
constexpr int kAdaOffBarriers = 0;                // full[32], empty[32]
constexpr int kAdaOffAbort = 512;
constexpr int kAdaOffStageRow = 576;              // [32] int64: the row a stage holds (-1: no more rows)
constexpr int kAdaOffGroupPos = 832;              // producer's ring bookkeeping (rings.cuh), 192 B
static_assert(kAdaOffGroupPos + kRingPosBytes <= 1024 && kAdaMaxGroups <= kRingMaxGroups, "shared memory map");
// per group: two row-parity buffers of [3][kAdaMaxWarps] floats (two sums, ok flags)
constexpr int kAdaOffPartial = 1024;
constexpr int kAdaPartialFloats = 2 * 3 * kAdaMaxWarps;
constexpr int kAdaOffStage0 = kAdaOffPartial + kAdaMaxGroups * kAdaPartialFloats * 4;   // 4096
constexpr int kAdaStageAlign = 128;

struct AdaLNParams {
  const char* x;
  char* out;
  long long x_stride, out_stride;                 // bytes per row
  long long tokens;
  long long rows_per_batch;
  const char* scale;
  const char* shift;
  long long mod_stride;                           // bytes between samples' rows
  int* status;
  unsigned long long wait_limit_ns;
  float eps;
  float inv_c;
  int hidden;                                     // C (multiple of 8)
  int consumer_warps;
  int group_warps;
  int stages;                                     // ring depth per group
  unsigned flags;
  unsigned row_bytes;                             // C * 2
  unsigned stage_bytes;
  unsigned smem_bytes;                            // dynamic shared memory of the launch
  int prefetch_rows;                              // first rows of the CTA prefetched into L2 before the wait
  // address spans of the buffers (checked builds test every access against them)
  MemSpan sp_x, sp_out, sp_scale, sp_shift;
};

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 8 modulation values of chunk k as fp32 pairs
template <typename MT>
__device__ __forceinline__ void load_mod8(const char* row, int k, float2 (&m)[4]);

template <>
__device__ __forceinline__ void load_mod8<float>(const char* row, int k, float2 (&m)[4]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(row) + 2 * k);
  const float4 b = __ldg(reinterpret_cast<const float4*>(row) + 2 * k + 1);
  m[0] = make_float2(a.x, a.y); m[1] = make_float2(a.z, a.w);
  m[2] = make_float2(b.x, b.y); m[3] = make_float2(b.z, b.w);
}

template <>
__device__ __forceinline__ void load_mod8<__nv_bfloat16>(const char* row, int k, float2 (&m)[4]) {
  Elem<__nv_bfloat16>::unpack(__ldg(reinterpret_cast<const uint4*>(row) + k), m);
}

template <>
__device__ __forceinline__ void load_mod8<__half>(const char* row, int k, float2 (&m)[4]) {
  Elem<__half>::unpack(__ldg(reinterpret_cast<const uint4*>(row) + k), m);
}

template <typename T, typename MT, int UNROLL>
__global__ void __launch_bounds__(kAdaMaxThreads, 1) adaln_kernel(const __grid_constant__ AdaLNParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NW = p.consumer_warps;
  const int GW = p.group_warps;
  const int n_groups = NW / GW;
  const int S = p.stages;
  const uint32_t base = smem_addr(smem);
  const uint32_t full0 = base + kAdaOffBarriers;
  const uint32_t empty0 = base + kAdaOffBarriers + 8 * kAdaMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAdaOffAbort);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S * n_groups; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, GW);
    }
    GroupRings(smem + kAdaOffGroupPos, n_groups, S, empty0).init();
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // All global memory accesses come after the previous kernel in the stream
  // has completed (programmatic dependent launch; see the QK kernel).  Only
  // L2 prefetches of the CTA's first p.prefetch_rows rows of x go before the
  // wait: they deliver no data, and the copies after the wait that hit them
  // see the previous kernel's writes.
  if (!kChecked && warp == NW && lane == 0) {
    long long row = blockIdx.x;
    for (int i = 0; i < p.prefetch_rows && row < p.tokens; ++i, row += gridDim.x)
      bulk_prefetch_l2(p.x + row * p.x_stride, p.row_bytes);
  }
  grid_dependency_wait();
  const unsigned long long limit = p.wait_limit_ns;

  if (warp == NW) {
    // ---------------- producer: one lane, one bulk copy per row
    if (lane != 0) return;
    const uint32_t stage0 = base + kAdaOffStage0;
    long long* stage_row = reinterpret_cast<long long*>(smem + kAdaOffStageRow);
    GroupRings rings(smem + kAdaOffGroupPos, n_groups, S, empty0);
    const long long step = gridDim.x;
    unsigned long long src = reinterpret_cast<unsigned long long>(p.x) + blockIdx.x * p.x_stride;
    const unsigned long long src_step = step * p.x_stride;
    bool ok = true;
    for (long long row = blockIdx.x; row < p.tokens; row += step) {
      const int gg = rings.free_group(limit, abort_flag, p.status);
      if (gg < 0) {
        ok = false;
        break;
      }
      if (p.flags & 1u) break;                    // test only: issue nothing
      const int s = gg * S + rings.slot(gg);
      // checked builds: the row inside x and the stage inside the launch's
      // shared memory, else nothing more is issued and the CTA gives up
      if (!in_span(reinterpret_cast<const void*>(src), p.row_bytes, p.sp_x, p.status) ||
          (kChecked && stage0 + (s + 1) * p.stage_bytes > base + p.smem_bytes)) {
        if (p.status) atomicCAS(p.status, 0, kStatusBounds);
        *abort_flag = 1;
        ok = false;
        break;
      }
      stage_row[s] = row;                         // published by the arrive below
      const uint32_t full = full0 + 8 * s;
      mbar_arrive_expect_tx(full, p.row_bytes);
      bulk_load(stage0 + s * p.stage_bytes, reinterpret_cast<const void*>(src), p.row_bytes, full);
      rings.advance(gg);
      src += src_step;
    }
    grid_dependents_launch();
    if (ok && !(p.flags & 1u)) {
      // no more rows: each group's next stage carries the end mark
      for (int done = 0; done < n_groups; ++done) {
        const int gg = rings.free_group(limit, abort_flag, p.status);
        if (gg < 0) {
          ok = false;
          break;
        }
        const int s = gg * S + rings.slot(gg);
        stage_row[s] = -1;
        mbar_arrive(full0 + 8 * s);
        rings.mark(gg);
      }
    }
    if (!ok || *abort_flag) rings.drain(full0, limit);
    return;
  }

  // ---------------- consumer warps
  const int grp = warp / GW, gw = warp % GW;
  const int gthreads = GW * 32;
  const int bar_id = 1 + grp;
  float* part_base = reinterpret_cast<float*>(smem + kAdaOffPartial) + grp * kAdaPartialFloats;
  const int n_chunks = p.hidden / 8;
  const int lane_g = gw * 32 + lane;
  const float eps = p.eps, inv_c = p.inv_c;
  // values this thread sums per row: chunks lane_g, lane_g + gthreads, ...
  const float my_n = lane_g < n_chunks ? 8.0f * static_cast<float>((n_chunks - 1 - lane_g) / gthreads + 1) : 0.0f;
  const int ring0 = grp * S;

  const long long* stage_row = reinterpret_cast<const long long*>(smem + kAdaOffStageRow);
  int s = 0;
  uint32_t ph = 0;
  int parity = 0;                                 // partial-sum buffer of this row
  for (;;) {
    const uint32_t full = full0 + 8 * (ring0 + s);
    const bool got = mbar_try_wait(full, ph) || bounded_wait(full, ph, limit, abort_flag, p.status);
    // the row this stage holds; the end mark (or a failed wait) makes the
    // group leave together at the barrier below
    const long long row = got ? stage_row[ring0 + s] : -1;
    const bool ok = got && row >= 0;
    const long long batch = ok ? row / p.rows_per_batch : 0;
    const unsigned char* st = smem + kAdaOffStage0 + (ring0 + s) * p.stage_bytes;

    float2 a1 = make_float2(0.0f, 0.0f), a2 = make_float2(0.0f, 0.0f);
    float k_minus_k0 = 0.0f, K = 0.0f;
    if (ok) {
      // one pass: sums of (x - k) and (x - k)^2, k = the first value of this
      // thread's first chunk
      float2 first[4], mine[4];
      Elem<T>::unpack(*reinterpret_cast<const uint4*>(st), first);
      K = shift_of_first8(first);
      float kt = 0.0f;
      if (lane_g < n_chunks) {
        Elem<T>::unpack(*reinterpret_cast<const uint4*>(st + lane_g * 16), mine);
        kt = mine[0].x;
      }
      k_minus_k0 = __fsub_rn(kt, K);
      const float2 nk = make_float2(-kt, -kt);
#pragma unroll UNROLL
      for (int k = lane_g; k < n_chunks; k += gthreads) {
        float2 X[4];
        Elem<T>::unpack(*reinterpret_cast<const uint4*>(st + k * 16), X);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 d = __fadd2_rn(X[j], nk);
          a1 = __fadd2_rn(a1, d);
          a2 = __ffma2_rn(d, d, a2);
        }
      }
    }
    const Moments wm = warp_moments(moments_of(my_n, k_minus_k0, __fadd_rn(a1.x, a1.y), __fadd_rn(a2.x, a2.y)),
                                    warp_count(gw, n_chunks, gthreads, 8));
    // post the warp's part and whether its wait succeeded.  Rows alternate
    // between two buffers: a warp can start the next row's posting while a
    // slower one still reads this row's parts, but cannot get two rows ahead
    // without passing the next row's barrier.
    float* part = part_base + parity * 3 * kAdaMaxWarps;
    parity ^= 1;
    if (lane == 0) {
      part[gw] = wm.u;
      part[kAdaMaxWarps + gw] = wm.m;
      part[2 * kAdaMaxWarps + gw] = ok ? 1.0f : 0.0f;
    }
    // this row's sample's modulation rows (the same for every row of the
    // sample: L1/L2 hits); their loads overlap the barrier
    const char* srow = p.scale + batch * p.mod_stride;
    const char* hrow = p.shift + batch * p.mod_stride;
    named_barrier(bar_id, gthreads);
    bool all_ok = true;
    const float ref = part[0];                    // warp 0 holds values whenever the row does
    RefSums sums;
    for (int w = 0; w < GW; ++w) {
      sums.add(Moments{warp_count(w, n_chunks, gthreads, 8), part[w], part[kAdaMaxWarps + w]}, ref);
      all_ok = all_ok && part[2 * kAdaMaxWarps + w] != 0.0f;
    }
    if (!all_ok) break;                           // every warp of the group leaves together
    // checked builds: the row's modulation rows and its output row inside
    // their buffers (the same answer in every warp of the group)
    const bool row_ok = in_span(srow, static_cast<unsigned long long>(p.hidden) * sizeof(MT), p.sp_scale, p.status) &&
                        in_span(hrow, static_cast<unsigned long long>(p.hidden) * sizeof(MT), p.sp_shift, p.status) &&
                        in_span(p.out + row * p.out_stride, p.row_bytes, p.sp_out, p.status);
    const Moments row_m = merged(static_cast<float>(p.hidden), ref, sums);
    const float m1 = row_m.u;                     // mean - K
    const float var = __fmul_rn(row_m.m, inv_c);
    const float r = rsqrtf(__fadd_rn(var, eps));
    const float2 R = make_float2(r, r);
    // normalise as (x - K) * r - m1 * r: x - K is exact for nearby values
    // and m1 = mean - K is rounded only to its own size, where x - (K + m1)
    // would carry the rounding of the mean itself, ulps of a small result
    // when |mean| is large against the spread
    const float2 nk = make_float2(-K, -K);
    const float c0 = __fmul_rn(-m1, r);
    const float2 C0 = make_float2(c0, c0);
    // second pass over the staged row: normalise, modulate, store
    char* orow = p.out + row * p.out_stride;
#pragma unroll UNROLL
    for (int k = row_ok ? lane_g : n_chunks; k < n_chunks; k += gthreads) {
      float2 X[4], sc[4], sh[4], o[4];
      Elem<T>::unpack(*reinterpret_cast<const uint4*>(st + k * 16), X);
      load_mod8<MT>(srow, k, sc);
      load_mod8<MT>(hrow, k, sh);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 sc1 = __fadd2_rn(sc[j], make_float2(1.0f, 1.0f));
        o[j] = __ffma2_rn(__ffma2_rn(__fadd2_rn(X[j], nk), R, C0), sc1, sh[j]);
      }
      store16(orow + k * 16, Elem<T>::pack(o));
    }
    // the row has been read for the last time: hand the stage back
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * (ring0 + s));
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
}

}  // namespace qknr
