// Fused DiT QK-RMSNorm + RoPE kernel for sm_103a.
//
// One persistent CTA per SM slot walks token rows t = blockIdx.x,
// blockIdx.x + gridDim.x, ...  A producer warp streams each row's Q and K
// heads (and V when it is copied), plus that row's cos and sin, from HBM
// into shared-memory stages with 1-D bulk copies (cp.async.bulk,
// completion counted on an mbarrier).  The consumer warps form groups; the
// CTA's rows go to the groups in turn and each group has its own ring of
// stages, which it drains strictly in order (so a group never waits on a
// stage phase more than one ahead of the barrier).  A group normalises and
// rotates every head of its row in fp32 registers, stores the result with
// 16-byte (interleaved) or 8-byte (rotate-half) stores and hands the stage
// back.
//
// Lane mapping: a lane owns 8 dimensions (16 bytes) of a head, so a head of
// D dims spans LPH = D/8 lanes and a warp covers HPW = 32/LPH heads at
// once.  With interleaved pairing lane j of a head owns the consecutive dims
// [8j, 8j+8) (one 16-byte access); with rotate-half pairing it owns
// [4j, 4j+4) and [D/2+4j, D/2+4j+4) (two 8-byte accesses), so in both
// styles every rotation partner sits in the same lane and the rotation
// needs no shuffle.  The per-head sum of squares is a shuffle-xor reduction
// inside the head's LPH lanes.  Consumer warps form groups
// that each take whole rows, so several rows are in flight at once; inside
// a group the warps are split between Q and K heads, so each folds only its
// own tensor's gain, and a warp works on two passes of heads at a time to
// overlap their latencies.
//
// cos/sin (page 1, "VisualGen Wan: deduplicate shared RoPE SMEM staging",
// Description): the shared layout stages one row per token and every head
// reads it by dimension.  Because a lane's dimensions are the same for
// every head it visits, each lane folds gamma and the staged cos/sin row
// into its coefficients a[d] = gamma[d]*cos[d], b[d] = s(d)*gamma[p(d)]*sin[d]
// once per row and reuses them for all heads.  The per-head expanded
// layout computes the same products per head from that head's table row;
// the operations are identical, so the two layouts give the same bits
// whenever their tables hold the same values (page 1, Test Coverage).
//
// Every mbarrier wait is bounded by a %globaltimer deadline.  When one
// runs out the CTA records QKNR_ERR_TIMEOUT in the caller's status word,
// raises a shared abort flag so its other warps stop waiting, waits
// (bounded) for the bulk copies it still has in flight, and returns.
#pragma once

#include "qknr_ptx.cuh"

namespace qknr {

constexpr int kMaxConsumerWarps = 16;
constexpr int kMaxThreads = 32 * (kMaxConsumerWarps + 1);
constexpr int kMaxStages = 32;        // all groups' rings together
// dynamic shared memory map (bytes)
constexpr int kOffBarriers = 0;       // full[kMaxStages], empty[kMaxStages]: 8 B each
constexpr int kOffAbort = 512;        // int abort flag
constexpr int kOffGamma = 1024;       // gamma_q[D], gamma_k[D] fp32 (D <= 128)
constexpr int kOffStage0 = 2048;      // stage rings
constexpr int kStageAlign = 128;

constexpr unsigned kFlagTestStall = 1u;
constexpr unsigned kFlagNoOverlap = 2u;     // plain launch, no L2 prefetch before the wait

struct KernelParams {
  const char* q;
  const char* k;
  const char* v;
  char* q_out;
  char* k_out;
  char* v_out;
  long long q_stride, k_stride, v_stride;            // bytes per row
  long long q_out_stride, k_out_stride, v_out_stride;
  long long tokens;
  long long cos_rows;
  const char* cos;
  const char* sin;
  long long cos_row_bytes;                           // one cos (or sin) table row
  const float* gamma_q;
  const float* gamma_k;
  int* status;
  unsigned long long wait_limit_ns;
  float eps;
  float inv_d;
  int hq, hk, hv;                                    // hv: V heads copied (0: V untouched)
  int consumer_warps;
  int group_warps;                                   // warps that share one row (divides consumer_warps)
  int warps_q, warps_k;                              // warps of a group on Q heads / on K heads
  int stages;                                        // ring depth of each group (stages per group)
  int qk_merged;                                     // K directly follows Q: one copy for both
  unsigned flags;
  // stage layout: [Q heads | K heads | V heads | cos row | sin row]
  unsigned off_k, off_v, off_cos, off_sin;
  unsigned stage_bytes;                              // stride between stages
  unsigned tx_bytes;                                 // bytes landing per stage
  unsigned smem_bytes;                               // dynamic shared memory of the launch
  int prefetch_rows;                                 // rows of the second ring fill prefetched before the wait (0: none)
  // address spans of the buffers (checked builds test every access against them)
  MemSpan sp_q, sp_k, sp_v, sp_q_out, sp_k_out, sp_v_out, sp_cos, sp_sin, sp_gq, sp_gk;
};

// What a checked build tests one tensor's accesses of one row against: the
// row's stage in shared memory and the output buffer.
struct RowChecks {
  const unsigned char* stage;
  unsigned stage_bytes;
  MemSpan out;
  int* status;
};

// ---------------------------------------------------------------------------
// per-lane rotation geometry

template <int D, bool RH>
struct Geometry {
  static constexpr int LPH = D / 8;       // lanes per head
  static constexpr int HPW = 32 / LPH;    // heads per warp pass
  // first dimension of the lane's low and high group of four (j = lane
  // index within its head); interleaved: [8j, 8j+8), rotate-half: [4j, 4j+4)
  // and its partners [D/2+4j, D/2+4j+4)
  static __device__ __forceinline__ int lo(int j) { return RH ? 4 * j : 8 * j; }
  static __device__ __forceinline__ int hi(int j) { return RH ? D / 2 + 4 * j : 8 * j + 4; }
};

// The lane's 8 activation values of one head (16 bytes at `head` + lo and
// + hi elements; one access when they are adjacent).
template <bool RH>
__device__ __forceinline__ uint4 load_lane8(const unsigned char* head, int lo, int hi) {
  if (!RH) return *reinterpret_cast<const uint4*>(head + lo * 2);
  const uint2 a = *reinterpret_cast<const uint2*>(head + lo * 2);
  const uint2 b = *reinterpret_cast<const uint2*>(head + hi * 2);
  return make_uint4(a.x, a.y, b.x, b.y);
}

template <bool RH>
__device__ __forceinline__ void store_lane8(char* head, int lo, int hi, const uint4& v) {
  if (!RH) {
    store16(head + lo * 2, v);
  } else {
    store8(head + lo * 2, make_uint2(v.x, v.y));
    store8(head + hi * 2, make_uint2(v.z, v.w));
  }
}

// The lane's 8 cos (or sin) values of one table row, widened to fp32 pairs.
template <typename CT, bool RH>
__device__ __forceinline__ void load_table_lane(const unsigned char* row, int lo, int hi, float2 (&c)[4]) {
  constexpr int CES = sizeof(CT);
  if (!RH) {
    load_table8<CT>(row + lo * CES, c);
  } else {
    float2 a[2], b[2];
    load_table4<CT>(row + lo * CES, a);
    load_table4<CT>(row + hi * CES, b);
    c[0] = a[0]; c[1] = a[1]; c[2] = b[0]; c[3] = b[1];
  }
}

// a[d] = g[d]*c[d]; b[d] = s(d) * g[p(d)] * s[d]  (each product rounded in fp32),
// held as pairs A[i] for the lane's elements 2i, 2i+1 (see Geometry).
// gamma points at the tensor's gains in shared memory.
template <int D, bool RH>
__device__ __forceinline__ void fold_coefficients(const float* gamma, int lo, int hi, const float2 (&C)[4],
                                                  const float2 (&Sn)[4], float2 (&A)[4], float2 (&B)[4]) {
  const float4 g0 = *reinterpret_cast<const float4*>(gamma + lo);
  const float4 g1 = *reinterpret_cast<const float4*>(gamma + hi);
  const float2 G[4] = {make_float2(g0.x, g0.y), make_float2(g0.z, g0.w), make_float2(g1.x, g1.y),
                       make_float2(g1.z, g1.w)};
  // gains of the rotation partners: the other group of four (rotate-half),
  // the other member of the same pair (interleaved)
  float2 GP[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) GP[i] = RH ? G[i ^ 2] : make_float2(G[i].y, G[i].x);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    A[i] = __fmul2_rn(G[i], C[i]);
    const float2 t = __fmul2_rn(GP[i], Sn[i]);
    // first pair members take -partner*sin: the lower half (rotate-half),
    // even dims (interleaved)
    if (RH)
      B[i] = i < 2 ? make_float2(-t.x, -t.y) : t;
    else
      B[i] = make_float2(-t.x, t.y);
  }
}

// Normalise and rotate the 8 elements this lane holds of one head (raw
// storage in `raw`, element order of Geometry), giving fp32 outputs O[i]
// for elements 2i, 2i+1.  Every lane of the warp must call it: the
// reduction shuffles the warp.
template <typename T, int D, bool RH>
__device__ __forceinline__ void head_math(const uint4& raw, const float2 (&A)[4], const float2 (&B)[4],
                                          float eps, float inv_d, float2 (&O)[4]) {
  constexpr int LPH = Geometry<D, RH>::LPH;
  float2 X[4];
  Elem<T>::unpack(raw, X);
  // sum of squares: even and odd elements in two fixed-order chains, then a
  // butterfly over the head's lanes
  float2 S2 = __fmul2_rn(X[0], X[0]);
  S2 = __ffma2_rn(X[1], X[1], S2);
  S2 = __ffma2_rn(X[2], X[2], S2);
  S2 = __ffma2_rn(X[3], X[3], S2);
  float ss = __fadd_rn(S2.x, S2.y);
#pragma unroll
  for (int off = LPH / 2; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
  const float r = rsqrtf(__fmaf_rn(ss, inv_d, eps));
  const float2 R = make_float2(r, r);
  // XP[i] holds the rotation partners of X[i], all in this lane
  float2 XP[4];
  if (RH) {
#pragma unroll
    for (int i = 0; i < 4; ++i) XP[i] = X[i ^ 2];
  } else {
    Elem<T>::unpack_swapped(raw, XP);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) O[i] = __fmul2_rn(__ffma2_rn(X[i], A[i], __fmul2_rn(XP[i], B[i])), R);
}

// One tensor's heads of one staged row: this warp takes passes
// lw, lw + G, lw + 2G, ... (a pass = HPW heads), two at a time so the
// latencies of one pass hide behind the other's.
template <typename T, typename CT, int D, bool RH, bool EXPANDED>
__device__ __forceinline__ void process_tensor(const unsigned char* seg, const unsigned char* cos_s,
                                               const unsigned char* sin_s, const float* gamma, char* out_row,
                                               int n_heads, int n_pass, int lw, int G, int lane, float eps,
                                               float inv_d, const RowChecks& ck) {
  using Geo = Geometry<D, RH>;
  constexpr int LPH = Geo::LPH;
  constexpr int HPW = Geo::HPW;
  constexpr int ES = 2;
  constexpr int CES = sizeof(CT);
  const int lo = Geo::lo(lane % LPH), hi = Geo::hi(lane % LPH);
  const int hslot = lane / LPH;
  // checked builds: head 0's staged values and the shared table row (read
  // by every lane, also for heads past the last) must lie in the stage; a
  // head whose own staged values, table row or output fall outside is
  // skipped (warp-uniform for the first test, per lane for the second)
  if (!in_smem(seg, D * ES, ck.stage, ck.stage_bytes, ck.status) ||
      !in_smem(cos_s, D * CES, ck.stage, ck.stage_bytes, ck.status) ||
      !in_smem(sin_s, D * CES, ck.stage, ck.stage_bytes, ck.status))
    return;
  auto head_ok = [&](int h) {
    bool ok = in_smem(seg + h * D * ES, D * ES, ck.stage, ck.stage_bytes, ck.status);
    if (EXPANDED)
      ok = ok && in_smem(cos_s + h * D * CES, D * CES, ck.stage, ck.stage_bytes, ck.status) &&
           in_smem(sin_s + h * D * CES, D * CES, ck.stage, ck.stage_bytes, ck.status);
    return ok && in_span(out_row + h * D * ES, D * ES, ck.out, ck.status);
  };
  float2 a[4], b[4];
  if (!EXPANDED) {
    // the row's one cos/sin row, folded once for every head this lane visits
    float2 c[4], s[4];
    load_table_lane<CT, RH>(cos_s, lo, hi, c);
    load_table_lane<CT, RH>(sin_s, lo, hi, s);
    fold_coefficients<D, RH>(gamma, lo, hi, c, s, a, b);
  }
  int t = lw;
  for (; t + G < n_pass; t += 2 * G) {
    const int h0 = t * HPW + hslot;
    const int h1 = (t + G) * HPW + hslot;
    const bool act0 = h0 < n_heads && head_ok(h0), act1 = h1 < n_heads && head_ok(h1);
    const int hc0 = act0 ? h0 : 0, hc1 = act1 ? h1 : 0;
    const uint4 r0 = load_lane8<RH>(seg + hc0 * D * ES, lo, hi);
    const uint4 r1 = load_lane8<RH>(seg + hc1 * D * ES, lo, hi);
    float2 o0[4], o1[4];
    if (EXPANDED) {
      float2 c[4], s[4], a1[4], b1[4];
      load_table_lane<CT, RH>(cos_s + hc0 * D * CES, lo, hi, c);
      load_table_lane<CT, RH>(sin_s + hc0 * D * CES, lo, hi, s);
      fold_coefficients<D, RH>(gamma, lo, hi, c, s, a, b);
      load_table_lane<CT, RH>(cos_s + hc1 * D * CES, lo, hi, c);
      load_table_lane<CT, RH>(sin_s + hc1 * D * CES, lo, hi, s);
      fold_coefficients<D, RH>(gamma, lo, hi, c, s, a1, b1);
      head_math<T, D, RH>(r0, a, b, eps, inv_d, o0);
      head_math<T, D, RH>(r1, a1, b1, eps, inv_d, o1);
    } else {
      head_math<T, D, RH>(r0, a, b, eps, inv_d, o0);
      head_math<T, D, RH>(r1, a, b, eps, inv_d, o1);
    }
    if (act0) store_lane8<RH>(out_row + h0 * D * ES, lo, hi, Elem<T>::pack(o0));
    if (act1) store_lane8<RH>(out_row + h1 * D * ES, lo, hi, Elem<T>::pack(o1));
  }
  if (t < n_pass) {
    const int h0 = t * HPW + hslot;
    const bool act0 = h0 < n_heads && head_ok(h0);
    const int hc0 = act0 ? h0 : 0;
    const uint4 r0 = load_lane8<RH>(seg + hc0 * D * ES, lo, hi);
    if (EXPANDED) {
      float2 c[4], s[4];
      load_table_lane<CT, RH>(cos_s + hc0 * D * CES, lo, hi, c);
      load_table_lane<CT, RH>(sin_s + hc0 * D * CES, lo, hi, s);
      fold_coefficients<D, RH>(gamma, lo, hi, c, s, a, b);
    }
    float2 o0[4];
    head_math<T, D, RH>(r0, a, b, eps, inv_d, o0);
    if (act0) store_lane8<RH>(out_row + h0 * D * ES, lo, hi, Elem<T>::pack(o0));
  }
}

// ---------------------------------------------------------------------------
// L2 prefetch of the CTA's second ring fill: with n = p.prefetch_rows (the
// rows of all its groups' rings), rows blockIdx.x + (n + i) * gridDim.x for
// i < n, every segment the producer will copy for them.  The first fill is
// left to the producer's own copies, which go out at once after the wait;
// the prefetched rows are then in L2 when the stages free up.

template <int D>
__device__ __forceinline__ void prefetch_second_fill(const KernelParams& p) {
  constexpr int ES = 2;
  const uint32_t q_bytes = p.hq * D * ES, k_bytes = p.hk * D * ES, v_bytes = p.hv * D * ES;
  const uint32_t c_bytes = static_cast<uint32_t>(p.cos_row_bytes);
  const int n = p.prefetch_rows;
  long long row = blockIdx.x + static_cast<long long>(n) * gridDim.x;
  for (int i = 0; i < n && row < p.tokens; ++i, row += gridDim.x) {
    if (p.qk_merged) {
      bulk_prefetch_l2(p.q + row * p.q_stride, q_bytes + k_bytes);
    } else {
      if (q_bytes) bulk_prefetch_l2(p.q + row * p.q_stride, q_bytes);
      if (k_bytes) bulk_prefetch_l2(p.k + row * p.k_stride, k_bytes);
    }
    if (v_bytes) bulk_prefetch_l2(p.v + row * p.v_stride, v_bytes);
    if (c_bytes) {
      const long long crow = row % p.cos_rows;
      bulk_prefetch_l2(p.cos + crow * p.cos_row_bytes, c_bytes);
      bulk_prefetch_l2(p.sin + crow * p.cos_row_bytes, c_bytes);
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel

template <typename T, typename CT, int D, bool RH, bool EXPANDED>
__global__ void __launch_bounds__(kMaxThreads, 1) qknr_fused_kernel(const __grid_constant__ KernelParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Geo = Geometry<D, RH>;
  constexpr int HPW = Geo::HPW;
  constexpr int ES = 2;                      // activation bytes

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  const int NW = p.consumer_warps;
  const uint32_t base = smem_addr(smem);
  const uint32_t full0 = base + kOffBarriers;
  const uint32_t empty0 = base + kOffBarriers + 8 * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  float* gam = reinterpret_cast<float*>(smem + kOffGamma);   // [0,D): gamma_q, [D,2D): gamma_k

  if (threadIdx.x == 0) {
    for (int s = 0; s < S * (NW / p.group_warps); ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, p.group_warps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Nothing above touches global memory, so under programmatic dependent
  // launch it overlaps the end of the kernel before this one in the stream.
  // Every global read and write comes after this wait: the inputs may be
  // that kernel's outputs, and an in-place output may be its input.  Only
  // L2 prefetches go before it (when the launch asks for them): they read
  // nothing into the CTA, and a load after the wait that hits a prefetched
  // line sees what the previous kernel wrote (its writes reach the same L2
  // lines), so those rows' DRAM reads overlap that kernel's last rows.
  if (!kChecked && p.prefetch_rows && warp == NW && lane == 0 && !(p.flags & kFlagNoOverlap))
    prefetch_second_fill<D>(p);
  grid_dependency_wait();

  const unsigned long long limit = p.wait_limit_ns;

  if (warp == NW) {
    // ---------------- producer warp: one lane issues every bulk copy
    if (lane != 0) return;
    const uint32_t q_bytes = p.hq * D * ES, k_bytes = p.hk * D * ES, v_bytes = p.hv * D * ES;
    const uint32_t c_bytes = static_cast<uint32_t>(p.cos_row_bytes);
    const uint32_t stage0 = base + kOffStage0;
    const int n_groups = NW / p.group_warps;
    // Row `issued` of this CTA goes to group g = issued % n_groups, slot
    // j % S of that group's ring with phase (j / S) & 1, where j counts the
    // group's rows.  All of it is kept as running counters: this one thread
    // issues every copy of the CTA, so its per-row cost bounds the rate.
    long long issued = 0;
    int g = 0, js = 0;
    uint32_t ph = 0;
    const long long step = gridDim.x;
    const long long crow_step = step % p.cos_rows;
    long long crow = blockIdx.x % p.cos_rows;
    // source addresses as integers: unused tensors may have null bases
    unsigned long long qsrc = reinterpret_cast<unsigned long long>(p.q) + blockIdx.x * p.q_stride;
    unsigned long long ksrc = reinterpret_cast<unsigned long long>(p.k) + blockIdx.x * p.k_stride;
    unsigned long long vsrc = reinterpret_cast<unsigned long long>(p.v) + blockIdx.x * p.v_stride;
    const unsigned long long qstep = step * p.q_stride, kstep = step * p.k_stride, vstep = step * p.v_stride;
    bool ok = true;
    for (long long row = blockIdx.x; row < p.tokens; row += step) {
      const int s = g * S + js;
      const uint32_t empty = empty0 + 8 * s;
      if (!mbar_try_wait(empty, ph ^ 1u) && !bounded_wait(empty, ph ^ 1u, limit, abort_flag, p.status)) {
        ok = false;
        break;
      }
      if (p.flags & kFlagTestStall) break;   // issue nothing: the consumers' waits run out
      const uint32_t full = full0 + 8 * s;
      const uint32_t dst = stage0 + s * p.stage_bytes;
      // checked builds: every source inside its buffer and the stage inside
      // the launch's shared memory; a copy that fails is not issued (its
      // stage then never completes and the waits on it run out)
      const void* qp = reinterpret_cast<const void*>(qsrc);
      const void* kp = reinterpret_cast<const void*>(ksrc);
      const void* vp = reinterpret_cast<const void*>(vsrc);
      const char* cp = p.cos + crow * p.cos_row_bytes;
      const char* sp = p.sin + crow * p.cos_row_bytes;
      const bool ok_copy = (!kChecked || dst + p.tx_bytes <= base + p.smem_bytes) &&
                           (!q_bytes || in_span(qp, q_bytes, p.sp_q, p.status)) &&
                           (!k_bytes || in_span(p.qk_merged ? static_cast<const char*>(qp) + q_bytes : kp, k_bytes,
                                                p.sp_k, p.status)) &&
                           (!v_bytes || in_span(vp, v_bytes, p.sp_v, p.status)) &&
                           (!c_bytes || (in_span(cp, c_bytes, p.sp_cos, p.status) &&
                                         in_span(sp, c_bytes, p.sp_sin, p.status)));
      if (!ok_copy) {
        if (p.status) atomicCAS(p.status, 0, kStatusBounds);
        *abort_flag = 1;
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(full, p.tx_bytes);
      if (p.qk_merged) {
        bulk_load(dst, qp, q_bytes + k_bytes, full);
      } else {
        if (q_bytes) bulk_load(dst, qp, q_bytes, full);
        if (k_bytes) bulk_load(dst + p.off_k, kp, k_bytes, full);
      }
      if (v_bytes) bulk_load(dst + p.off_v, vp, v_bytes, full);
      if (c_bytes) {
        bulk_load(dst + p.off_cos, cp, c_bytes, full);
        bulk_load(dst + p.off_sin, sp, c_bytes, full);
      }
      ++issued;
      qsrc += qstep;
      ksrc += kstep;
      vsrc += vstep;
      crow += crow_step;
      if (crow >= p.cos_rows) crow -= p.cos_rows;
      if (++g == n_groups) {
        g = 0;
        if (++js == S) {
          js = 0;
          ph ^= 1u;
        }
      }
    }
    // every load of this CTA is issued: the next kernel in the stream may
    // start launching (its CTAs take an SM as this grid's CTAs leave it)
    grid_dependents_launch();
    if (!ok || *abort_flag) {
      // copies of the last n_groups * S issued rows (the latest use of every
      // stage) may still be landing: wait for them before this CTA's shared
      // memory is released
      const long long total = static_cast<long long>(n_groups) * S;
      const long long first = issued > total ? issued - total : 0;
      for (long long it = first; it < issued; ++it) {
        const long long j = it / n_groups;
        const uint32_t bar = full0 + 8 * (static_cast<int>(it % n_groups) * S + static_cast<int>(j % S));
        const uint32_t phase = static_cast<uint32_t>((j / S) & 1);
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(bar, phase) && global_timer_ns() - t0 < limit) {
        }
      }
    }
    return;
  }

  // ---------------- consumer warps
  // The gains go to shared memory while the producer's first loads are in
  // flight; the consumer warps alone wait for them (named barrier 1).
  for (int i = threadIdx.x; i < 2 * D; i += NW * 32) {
    // a tensor with no heads may come without its gains: not read then
    const float* g = i < D ? (p.hq ? p.gamma_q : nullptr) : (p.hk ? p.gamma_k : nullptr);
    const float* gi = g ? g + (i < D ? i : i - D) : nullptr;
    gam[i] = gi && in_span(gi, 4, i < D ? p.sp_gq : p.sp_gk, p.status) ? *gi : 1.0f;
  }
  named_barrier_sync(1, NW * 32);

  // The consumer warps form NW / GW groups of GW warps; group g takes the
  // CTA's rows g, g + NW/GW, ... so several rows are in flight at once.
  // Inside a group, warps [0, warps_q) normalise Q heads and warps
  // [GW - warps_k, GW) K heads (disjoint unless GW == 1); all of the
  // group's warps share the V copy.
  const int GW = p.group_warps;
  const int n_groups = NW / GW;
  const int grp = warp / GW, gw = warp % GW;
  const int nq = (p.hq + HPW - 1) / HPW;                // Q passes per row
  const int nk = (p.hk + HPW - 1) / HPW;                // K passes per row
  const int v_row = p.hv * D * ES;                      // V bytes per row
  const bool do_q = gw < p.warps_q;
  const bool do_k = gw >= GW - p.warps_k;
  const float eps = p.eps, inv_d = p.inv_d;

  const int ring0 = grp * S;                            // this group's ring
  int s = 0;
  uint32_t ph = 0;
  for (long long row = blockIdx.x + static_cast<long long>(grp) * gridDim.x; row < p.tokens;
       row += static_cast<long long>(n_groups) * gridDim.x) {
    const uint32_t full = full0 + 8 * (ring0 + s);
    if (!mbar_try_wait(full, ph) && !bounded_wait(full, ph, limit, abort_flag, p.status)) break;
    const unsigned char* st = smem + kOffStage0 + (ring0 + s) * p.stage_bytes;
    if (do_q && nq)
      process_tensor<T, CT, D, RH, EXPANDED>(st, st + p.off_cos, st + p.off_sin, gam,
                                             p.q_out + row * p.q_out_stride, p.hq, nq, gw, p.warps_q, lane, eps,
                                             inv_d, RowChecks{st, p.stage_bytes, p.sp_q_out, p.status});
    if (do_k && nk)
      process_tensor<T, CT, D, RH, EXPANDED>(st + p.off_k, st + p.off_cos, st + p.off_sin, gam + D,
                                             p.k_out + row * p.k_out_stride, p.hk, nk, gw - (GW - p.warps_k),
                                             p.warps_k, lane, eps, inv_d,
                                             RowChecks{st, p.stage_bytes, p.sp_k_out, p.status});
    // V pass-through copy, 16 bytes per lane
    for (int off = (gw * 32 + lane) * 16; off < v_row; off += GW * 512) {
      const unsigned char* src = st + p.off_v + off;
      char* dstv = p.v_out + row * p.v_out_stride + off;
      if (in_smem(src, 16, st, p.stage_bytes, p.status) && in_span(dstv, 16, p.sp_v_out, p.status))
        store16(dstv, *reinterpret_cast<const uint4*>(src));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * (ring0 + s));
    if (++s == S) { s = 0; ph ^= 1u; }
  }
}

}  // namespace qknr
