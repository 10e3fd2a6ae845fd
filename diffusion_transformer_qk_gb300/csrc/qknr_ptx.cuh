// PTX helpers shared by the library's kernels (sm_100 family): mbarriers,
// 1-D bulk copies into shared memory, %globaltimer-bounded waits, streaming
// stores and 16-byte <-> fp32-pair conversions of bf16/fp16 storage.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qknr {

constexpr int kStatusTimeout = 6;     // QKNR_ERR_TIMEOUT
constexpr int kStatusBounds = 9;      // QKNR_ERR_BOUNDS

// ---------------------------------------------------------------------------
// Debug builds (QKNR_CHECKED): every global access is checked against the
// address span of the buffer it belongs to, and every shared-memory stage
// read against its stage.  An access outside them is skipped and
// QKNR_ERR_BOUNDS goes to the caller's status word (no assert, no trap).
// In the regular build the checks are constant true and compile away.

#ifdef QKNR_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// [lo, hi) byte addresses of a buffer (empty: lo == hi)
struct MemSpan {
  unsigned long long lo, hi;
};

__device__ __forceinline__ bool in_span(const void* p, unsigned long long bytes, const MemSpan& s, int* status) {
  if (!kChecked) return true;
  const unsigned long long a = reinterpret_cast<unsigned long long>(p);
  if (a >= s.lo && a + bytes >= a && a + bytes <= s.hi) return true;
  if (status) atomicCAS(status, 0, kStatusBounds);
  return false;
}

// a generic pointer into this CTA's shared memory, within [lo, lo + size)
__device__ __forceinline__ bool in_smem(const void* p, unsigned bytes, const void* lo, unsigned size, int* status) {
  if (!kChecked) return true;
  const char* a = static_cast<const char*>(p);
  const char* b = static_cast<const char*>(lo);
  if (a >= b && a + bytes <= b + size) return true;
  if (status) atomicCAS(status, 0, kStatusBounds);
  return false;
}

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

// The same test, but a thread whose phase is not complete is suspended
// (issuing nothing) until it completes or about `hint_ns` have passed.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialization may start while the kernel before it in the stream
// is still finishing; grid_dependency_wait() returns once that kernel has
// completed and its memory operations are visible (at once when there is no
// such kernel).  grid_dependents_launch() lets the kernel after this one
// start launching once every CTA of this grid has issued it or exited.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// bar.sync on a named barrier for `threads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted in
// bytes on `bar`.  Both addresses 16-byte aligned, bytes a multiple of 16.
// The source is marked evict-first in L2: every byte is streamed once.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Bring `bytes` at `src` into L2.  A hint: no data reaches the program, so
// it cannot observe a stale value (L2 is where every SM's writes land).
// 16-byte aligned address, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Wait for phase `parity` of `bar` to complete, giving up at the deadline
// or when another warp of the CTA has aborted.  Returns false on give-up.
// The waiting thread sleeps in the barrier (20 us at a time) instead of
// spinning, so waiters leave the issue slots to the warps doing work.
static __device__ __noinline__ bool bounded_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns, volatile int* abort_flag,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      if (status) atomicCAS(status, 0, kStatusTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// element conversions: 16 bytes of storage <-> 4 fp32 pairs (elements 2i, 2i+1)
// Arithmetic runs on Blackwell's paired fp32 instructions (__ffma2_rn and
// friends), each half rounded exactly as the scalar instruction would.

template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  // X[i] = (x[2i], x[2i+1])
  static __device__ __forceinline__ void unpack(const uint4& r, float2 (&X)[4]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) X[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
  // X[i] = (x[2i+1], x[2i])
  static __device__ __forceinline__ void unpack_swapped(const uint4& r, float2 (&X)[4]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) X[i] = make_float2(__uint_as_float(w[i] & 0xffff0000u), __uint_as_float(w[i] << 16));
  }
  static __device__ __forceinline__ uint4 pack(const float2 (&O)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(O[i].x, O[i].y);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Elem<__half> {
  static __device__ __forceinline__ void unpack(const uint4& r, float2 (&X)[4]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) X[i] = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
  }
  static __device__ __forceinline__ void unpack_swapped(const uint4& r, float2 (&X)[4]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      X[i] = make_float2(__high2float(h), __low2float(h));
    }
  }
  static __device__ __forceinline__ uint4 pack(const float2 (&O)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = __floats2half2_rn(O[i].x, O[i].y);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// 8 consecutive cos (or sin) values from shared memory, widened to fp32 pairs.
template <typename CT>
__device__ __forceinline__ void load_table8(const unsigned char* p, float2 (&c)[4]);

template <>
__device__ __forceinline__ void load_table8<float>(const unsigned char* p, float2 (&c)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 16);
  c[0] = make_float2(a.x, a.y); c[1] = make_float2(a.z, a.w);
  c[2] = make_float2(b.x, b.y); c[3] = make_float2(b.z, b.w);
}

template <>
__device__ __forceinline__ void load_table8<__nv_bfloat16>(const unsigned char* p, float2 (&c)[4]) {
  Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(p), c);
}

// 4 consecutive cos (or sin) values from shared memory, widened to fp32 pairs.
template <typename CT>
__device__ __forceinline__ void load_table4(const unsigned char* p, float2 (&c)[2]);

template <>
__device__ __forceinline__ void load_table4<float>(const unsigned char* p, float2 (&c)[2]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  c[0] = make_float2(a.x, a.y); c[1] = make_float2(a.z, a.w);
}

template <>
__device__ __forceinline__ void load_table4<__nv_bfloat16>(const unsigned char* p, float2 (&c)[2]) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  c[0] = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
  c[1] = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}


// 16- and 8-byte streaming stores to global memory (written once, not re-read).
__device__ __forceinline__ void store16(char* dst, const uint4& v) {
  __stcs(reinterpret_cast<uint4*>(dst), v);
}

__device__ __forceinline__ void store8(char* dst, const uint2& v) {
  __stcs(reinterpret_cast<uint2*>(dst), v);
}

}  // namespace qknr
