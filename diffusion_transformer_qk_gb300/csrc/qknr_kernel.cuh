// Fused DiT QK-RMSNorm + RoPE kernel for sm_103a.
//
// One persistent CTA per SM slot walks token rows t = blockIdx.x,
// blockIdx.x + gridDim.x, ...  A producer warp streams each row's Q and K
// heads (and V when it is copied), plus that row's cos and sin, from HBM
// into a ring of shared-memory stages with 1-D bulk copies
// (cp.async.bulk, completion counted on an mbarrier).  Consumer warps take
// a stage, normalise and rotate every head in fp32 registers and store the
// result with 16-byte stores, then hand the stage back.
//
// Lane mapping: a lane owns 8 consecutive dimensions (16 bytes) of a head,
// so a head of D dims spans LPH = D/8 lanes and a warp covers HPW = 32/LPH
// heads at once.  The per-head sum of squares is a shuffle-xor reduction
// inside those LPH lanes; a rotate-half partner lives in lane ^ (LPH/2),
// an interleaved partner in the same lane.
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

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qknr {

constexpr int kMaxConsumerWarps = 16;
constexpr int kMaxThreads = 32 * (kMaxConsumerWarps + 1);
constexpr int kMaxStages = 16;
// dynamic shared memory map (bytes)
constexpr int kOffBarriers = 0;       // full[kMaxStages], empty[kMaxStages]: 8 B each
constexpr int kOffAbort = 256;        // int abort flag
constexpr int kOffGamma = 512;        // gamma_q[D], gamma_k[D] fp32 (D <= 128)
constexpr int kOffStage0 = 1536;      // stage ring
constexpr int kStageAlign = 128;

constexpr int kStatusTimeout = 6;     // QKNR_ERR_TIMEOUT
constexpr unsigned kFlagTestStall = 1u;

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
  int stages;
  unsigned flags;
  // stage layout: [Q heads | K heads | V heads | cos row | sin row]
  unsigned off_k, off_v, off_cos, off_sin;
  unsigned stage_bytes;                              // stride between stages
  unsigned tx_bytes;                                 // bytes landing per stage
};

// ---------------------------------------------------------------------------
// PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted in
// bytes on `bar`.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void stg128(void* ptr, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Wait for phase `parity` of `bar` to complete, giving up at the deadline
// or when another warp of the CTA has aborted.  Returns false on give-up.
static __device__ __noinline__ bool bounded_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns, volatile int* abort_flag,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      if (status) atomicCAS(status, 0, kStatusTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// element conversions (16 bytes of storage <-> 8 fp32 values)

template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ void unpack(const uint4& r, float (&x)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ uint4 pack(const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Elem<__half> {
  static __device__ __forceinline__ void unpack(const uint4& r, float (&x)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 f = __half22float2(h);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = __floats2half2_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// 8 consecutive cos (or sin) values from shared memory, widened to fp32.
template <typename CT>
__device__ __forceinline__ void load_table8(uint32_t addr, float (&c)[8]);

template <>
__device__ __forceinline__ void load_table8<float>(uint32_t addr, float (&c)[8]) {
  const uint4 a = lds128(addr), b = lds128(addr + 16);
  c[0] = __uint_as_float(a.x); c[1] = __uint_as_float(a.y);
  c[2] = __uint_as_float(a.z); c[3] = __uint_as_float(a.w);
  c[4] = __uint_as_float(b.x); c[5] = __uint_as_float(b.y);
  c[6] = __uint_as_float(b.z); c[7] = __uint_as_float(b.w);
}

template <>
__device__ __forceinline__ void load_table8<__nv_bfloat16>(uint32_t addr, float (&c)[8]) {
  Elem<__nv_bfloat16>::unpack(lds128(addr), c);
}

// ---------------------------------------------------------------------------
// per-lane rotation geometry

template <int D, bool RH>
struct Geometry {
  static constexpr int LPH = D / 8;       // lanes per head
  static constexpr int HPW = 32 / LPH;    // heads per warp pass
  // dimension of the partner of element j of a lane starting at d0
  static __device__ __forceinline__ int partner_dim(int d0, int j) {
    return RH ? ((d0 + D / 2) % D) + j : d0 + (j ^ 1);
  }
  // true when element j of the lane is the first member of its pair
  static __device__ __forceinline__ bool first_member(int d0, int j) {
    return RH ? (d0 < D / 2) : ((j & 1) == 0);
  }
};

// a[j] = g[d]*c[j]; b[j] = s(d) * g[p(d)] * s[j]  (each product rounded in fp32)
template <int D, bool RH>
__device__ __forceinline__ void fold_coefficients(const float* gamma, int d0, const float (&c)[8],
                                                  const float (&s)[8], float (&a)[8],
                                                  float (&b)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float g = gamma[d0 + j];
    const float gp = gamma[Geometry<D, RH>::partner_dim(d0, j)];
    a[j] = __fmul_rn(g, c[j]);
    const float t = __fmul_rn(gp, s[j]);
    b[j] = Geometry<D, RH>::first_member(d0, j) ? -t : t;
  }
}

// Normalise and rotate the 8 elements this lane holds of one head (raw
// storage in `raw`), giving fp32 outputs in `o`.  Every lane of the warp
// must call it: the reductions and the partner exchange shuffle the warp.
template <typename T, int D, bool RH>
__device__ __forceinline__ void head_math(const uint4& raw, const float (&a)[8], const float (&b)[8],
                                          float eps, float inv_d, float (&o)[8]) {
  constexpr int LPH = Geometry<D, RH>::LPH;
  float x[8];
  Elem<T>::unpack(raw, x);
  // sum of squares: fixed order inside the lane, then a butterfly over the head's lanes
  float ss = __fmul_rn(x[0], x[0]);
#pragma unroll
  for (int j = 1; j < 8; ++j) ss = __fmaf_rn(x[j], x[j], ss);
#pragma unroll
  for (int off = LPH / 2; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
  const float r = rsqrtf(__fmaf_rn(ss, inv_d, eps));
  float xp[8];
  if (RH) {
    uint4 pr;
    pr.x = __shfl_xor_sync(0xffffffffu, raw.x, LPH / 2);
    pr.y = __shfl_xor_sync(0xffffffffu, raw.y, LPH / 2);
    pr.z = __shfl_xor_sync(0xffffffffu, raw.z, LPH / 2);
    pr.w = __shfl_xor_sync(0xffffffffu, raw.w, LPH / 2);
    Elem<T>::unpack(pr, xp);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) xp[j] = x[j ^ 1];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) o[j] = __fmul_rn(__fmaf_rn(x[j], a[j], __fmul_rn(xp[j], b[j])), r);
}

// ---------------------------------------------------------------------------
// the kernel

template <typename T, typename CT, int D, bool RH, bool EXPANDED>
__global__ void __launch_bounds__(kMaxThreads, 1) qknr_fused_kernel(const __grid_constant__ KernelParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  using G = Geometry<D, RH>;
  constexpr int LPH = G::LPH;
  constexpr int HPW = G::HPW;
  constexpr int ES = 2;                      // activation bytes
  constexpr int CES = sizeof(CT);            // table bytes

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  const uint32_t base = smem_addr(smem);
  const uint32_t full0 = base + kOffBarriers;
  const uint32_t empty0 = base + kOffBarriers + 8 * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  float* gam = reinterpret_cast<float*>(smem + kOffGamma);   // [0,D): gamma_q, [D,2D): gamma_k
  const uint32_t stage0 = base + kOffStage0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, p.consumer_warps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < 2 * D; i += blockDim.x) {
    const float* g = i < D ? p.gamma_q : p.gamma_k;
    gam[i] = g ? g[i < D ? i : i - D] : 1.0f;
  }
  __syncthreads();

  const unsigned long long limit = p.wait_limit_ns;

  if (warp == p.consumer_warps) {
    // ---------------- producer warp: one lane issues every bulk copy
    if (lane != 0) return;
    const uint32_t q_bytes = p.hq * D * ES, k_bytes = p.hk * D * ES, v_bytes = p.hv * D * ES;
    const uint32_t c_bytes = static_cast<uint32_t>(p.cos_row_bytes);
    long long issued = 0;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (long long row = blockIdx.x; row < p.tokens; row += gridDim.x) {
      if (!bounded_wait(empty0 + 8 * s, ph ^ 1u, limit, abort_flag, p.status)) { ok = false; break; }
      if (p.flags & kFlagTestStall) break;   // issue nothing: the consumers' waits run out
      const uint32_t full = full0 + 8 * s;
      const uint32_t dst = stage0 + s * p.stage_bytes;
      mbar_arrive_expect_tx(full, p.tx_bytes);
      if (q_bytes) bulk_load(dst, p.q + row * p.q_stride, q_bytes, full);
      if (k_bytes) bulk_load(dst + p.off_k, p.k + row * p.k_stride, k_bytes, full);
      if (v_bytes) bulk_load(dst + p.off_v, p.v + row * p.v_stride, v_bytes, full);
      if (c_bytes) {
        const long long crow = row % p.cos_rows;
        bulk_load(dst + p.off_cos, p.cos + crow * p.cos_row_bytes, c_bytes, full);
        bulk_load(dst + p.off_sin, p.sin + crow * p.cos_row_bytes, c_bytes, full);
      }
      ++issued;
      if (++s == S) { s = 0; ph ^= 1u; }
    }
    if (!ok || *abort_flag) {
      // copies of the last (up to S) issued stages may still be landing:
      // wait for them before this CTA's shared memory is released
      const long long first = issued > S ? issued - S : 0;
      for (long long it = first; it < issued; ++it) {
        const uint32_t bar = full0 + 8 * static_cast<int>(it % S);
        const uint32_t ph = static_cast<uint32_t>((it / S) & 1);
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(bar, ph) && global_timer_ns() - t0 < limit) {
        }
      }
    }
    return;
  }

  // ---------------- consumer warps
  const int sub = lane % LPH;           // lane's slot inside its head
  const int hslot = lane / LPH;         // which of the warp's HPW heads
  const int d0 = sub * 8;
  const int nq = (p.hq + HPW - 1) / HPW;                // Q passes per row
  const int nk = (p.hk + HPW - 1) / HPW;                // K passes per row
  const int nv = (p.hv * D * ES + 511) / 512;           // V copy passes (512 B per warp)
  const int ntask = nq + nk + nv;
  const float eps = p.eps, inv_d = p.inv_d;

  int s = 0;
  uint32_t ph = 0;
  for (long long row = blockIdx.x; row < p.tokens; row += gridDim.x) {
    if (!bounded_wait(full0 + 8 * s, ph, limit, abort_flag, p.status)) break;
    const uint32_t st = stage0 + s * p.stage_bytes;

    float aq[8], bq[8], ak[8], bk[8];
    if (!EXPANDED && nq + nk > 0) {
      // the row's shared cos/sin, read once by this lane for every head it visits
      float c[8], sn[8];
      load_table8<CT>(st + p.off_cos + d0 * CES, c);
      load_table8<CT>(st + p.off_sin + d0 * CES, sn);
      fold_coefficients<D, RH>(gam, d0, c, sn, aq, bq);
      fold_coefficients<D, RH>(gam + D, d0, c, sn, ak, bk);
    }

    for (int task = warp; task < ntask; task += p.consumer_warps) {
      if (task < nq + nk) {
        const bool is_k = task >= nq;
        const int h = (is_k ? task - nq : task) * HPW + hslot;   // head within its tensor
        const int nh = is_k ? p.hk : p.hq;
        const bool active = h < nh;
        const int hc = active ? h : 0;
        const uint32_t src = st + (is_k ? p.off_k : 0u) + (hc * D + d0) * ES;
        const uint4 raw = lds128(src);
        float a[8], b[8];
        if (EXPANDED) {
          float c[8], sn[8];
          load_table8<CT>(st + p.off_cos + (hc * D + d0) * CES, c);
          load_table8<CT>(st + p.off_sin + (hc * D + d0) * CES, sn);
          fold_coefficients<D, RH>(is_k ? gam + D : gam, d0, c, sn, a, b);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            a[j] = is_k ? ak[j] : aq[j];
            b[j] = is_k ? bk[j] : bq[j];
          }
        }
        float o[8];
        head_math<T, D, RH>(raw, a, b, eps, inv_d, o);
        if (active) {
          char* dst = is_k ? p.k_out + row * p.k_out_stride : p.q_out + row * p.q_out_stride;
          stg128(dst + (h * D + d0) * ES, Elem<T>::pack(o));
        }
      } else {
        // V pass-through copy, 16 bytes per lane
        const int off = (task - nq - nk) * 512 + lane * 16;
        if (off < p.hv * D * ES) {
          const uint4 raw = lds128(st + p.off_v + off);
          stg128(p.v_out + row * p.v_out_stride + off, raw);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (++s == S) { s = 0; ph ^= 1u; }
  }
}

}  // namespace qknr
