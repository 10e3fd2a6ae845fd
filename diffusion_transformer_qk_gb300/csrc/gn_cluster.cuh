// Group norm + SiLU with one thread-block cluster per group ("fused qknorm
// rope Flux 2.0", section "Not in this PR — follow-ups", names the VAE's
// group_norm_silu; the operation is restated in include/qknr_gn.h).
//
// When a group's (C/G)*H*W elements fit in the shared memory of a cluster
// of CTAs (up to 16 on GB300), the group is split into equal parts, one
// per CTA of its cluster.  Each CTA bulk-copies its part (and the group's
// first 16 bytes, whose lower median is the shift K) into shared memory,
// forms the part's statistics (the per-thread and per-warp merges of the
// two-pass statistics kernel, over the part instead of a piece), and
// leaves them in its shared memory.  After a cluster barrier every CTA
// reads all the parts' statistics of its cluster over distributed shared
// memory and merges them in one fixed order (the same in every CTA), so
// all of them hold the same mean and 1/sqrt(var + eps); then each writes
// silu((x - K)*a + b) for its own part from shared memory.  x is read
// once, there is no workspace, and no CTA waits for anything outside its
// own cluster, which the hardware schedules all at once.
//
// Every thread of every CTA of a cluster reaches both cluster barriers
// exactly once, whatever happens to its copy: a copy that does not land
// within the wait limit, or a part outside its buffer (checked builds),
// marks the CTA's part as unusable, the whole cluster then skips its
// writes, and a CTA whose copies may still be in flight waits for them
// (bounded) before it exits.
#pragma once

#include "gn_kernel.cuh"

namespace qknr {

constexpr int kGncMaxThreads = 1024;
constexpr int kGncOffFull = 0;                   // mbarrier of the part's copies
constexpr int kGncOffBad = 8;                    // int: this CTA's part is not usable
constexpr int kGncOffIssued = 12;                // int: the part's copies were issued
constexpr int kGncOffK = 16;                     // the group's first 16 bytes
constexpr int kGncOffPart = 32;                  // this CTA's part: mean - K, sum of squared deviations
constexpr int kGncOffCoef = 48;                  // m1, rstd, K, and 1.0 when the cluster skips its writes
constexpr int kGncOffRed = 64;                   // [2 * warps] floats
constexpr int kGncOffData = 384;                 // the part's elements
constexpr unsigned kGncCopyBytes = 32768;        // bytes per bulk copy
constexpr int kGncMaxCluster = 16;
static_assert(kGncOffRed + 8 * (kGncMaxThreads / 32) <= kGncOffData, "shared memory map");
static_assert(kGncOffData % 128 == 0, "shared memory map");

struct GnClusterParams {
  const char* x;
  char* out;
  const float* gamma;
  const float* beta;
  int* status;                 // optional
  long long span_len;          // L, elements of a group of one sample
  long long hw;                // H * W (a multiple of 8)
  long long part_len;          // elements per CTA of a cluster (a multiple of 8); the last part is shorter
  int groups;
  int group_channels;
  unsigned flags;
  unsigned smem_bytes;         // dynamic shared memory of the launch
  unsigned long long wait_limit_ns;
  float eps;
  // address spans of the buffers (checked builds test every access against them)
  MemSpan sp_x, sp_out, sp_gamma, sp_beta;
};

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ unsigned cluster_size() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ unsigned cluster_index() {
  unsigned r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// Cluster barrier, in two halves: every thread of every CTA of the cluster
// arrives (its earlier shared-memory writes released to the cluster), and
// a wait returns once all have arrived (acquiring what they released).
// Executed by whole warps.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A 32-bit word at shared-memory address `local` of CTA `rank` of this
// cluster (the same offset in that CTA's shared memory).
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t local, unsigned rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// The part of a CTA of NT threads from the threads' parts, as piece_moments
// (the same order for NT = 256): an xor tree in each warp, then thread 0
// merges the warps' parts in order.  Valid in thread 0.
template <int NT>
__device__ __forceinline__ Moments part_moments(const Moments& mine, int nvec, float* red) {
  constexpr int kWarps = NT / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Moments wp = warp_moments(mine, warp_count(warp, nvec, NT, 8));
  if (lane == 0) {
    red[warp] = wp.u;
    red[kWarps + warp] = wp.m;
  }
  __syncthreads();
  Moments t{0.0f, 0.0f, 0.0f};
  if (threadIdx.x == 0) {
    const float r = red[0];                      // warp 0 holds values whenever the part does
    RefSums sums;
    for (int w = 0; w < kWarps; ++w) sums.add(Moments{warp_count(w, nvec, NT, 8), red[w], red[kWarps + w]}, r);
    t = merged(8.0f * static_cast<float>(nvec), r, sums);
  }
  return t;
}

// Elements of part `rank` of a group of L elements in parts of `part`.
__device__ __forceinline__ long long part_elems(unsigned rank, long long part, long long L) {
  const long long lo = static_cast<long long>(rank) * part;
  const long long hi = lo + part < L ? lo + part : L;
  return hi > lo ? hi - lo : 0;
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT, 1) gn_cluster_kernel(const __grid_constant__ GnClusterParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = smem_addr(smem);
  const uint32_t full = base + kGncOffFull;
  volatile int* bad = reinterpret_cast<volatile int*>(smem + kGncOffBad);
  volatile int* issued = reinterpret_cast<volatile int*>(smem + kGncOffIssued);
  float* red = reinterpret_cast<float*>(smem + kGncOffRed);
  float* part = reinterpret_cast<float*>(smem + kGncOffPart);
  float* coef = reinterpret_cast<float*>(smem + kGncOffCoef);
  const unsigned rank = cluster_rank(), csize = cluster_size();
  const long long span = cluster_index();          // one group of one sample per cluster
  const long long L = p.span_len;
  const long long lo = static_cast<long long>(rank) * p.part_len;
  const int nvec = static_cast<int>(part_elems(rank, p.part_len, L) / 8);
  const unsigned bytes = static_cast<unsigned>(nvec) * 16u;
  const char* group = p.x + span * L * 2;

  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    *bad = 0;
    *issued = 0;
    fence_barrier_init();
    // the part and the group's first 16 bytes, counted on one barrier
    // (checked builds: both inside x and the part inside shared memory,
    // else nothing is issued and the part is unusable)
    const bool in_bounds = in_span(group, 16, p.sp_x, p.status) &&
                           (bytes == 0 || in_span(group + lo * 2, bytes, p.sp_x, p.status)) &&
                           (!kChecked || kGncOffData + bytes <= p.smem_bytes);
    if (!in_bounds) {
      if (p.status) atomicCAS(p.status, 0, kStatusBounds);
      *bad = 1;
    } else if (!(p.flags & kGnfFlagStallLoads)) {
      mbar_arrive_expect_tx(full, bytes + 16u);
      bulk_load(base + kGncOffK, group, 16u, full);
      for (unsigned off = 0; off < bytes; off += kGncCopyBytes)
        bulk_load(base + kGncOffData + off, group + lo * 2 + off, bytes - off < kGncCopyBytes ? bytes - off : kGncCopyBytes,
                  full);
      *issued = 1;
    }
  }
  __syncthreads();

  // every warp waits for the part (bounded; the test flag that issues no
  // copies makes this run out); one failure marks the part unusable
  bool got = false;
  if (!*bad) {
    if (lane == 0)
      got = mbar_try_wait_sleep(full, 0, kGnfSleepNs) ||
            bounded_wait(full, 0, p.wait_limit_ns, reinterpret_cast<volatile int*>(bad), p.status);
    got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
  }
  const bool ok = __syncthreads_and(got) != 0;

  // this part's statistics around K: thread t sums vectors t, t + NT, ...
  // in batches of kGnBatch around each batch's first value, as the two-pass
  // statistics kernel does over a piece
  float K = 0.0f;
  if (ok) {
    float2 first[4];
    Elem<T>::unpack(*reinterpret_cast<const uint4*>(smem + kGncOffK), first);
    K = shift_of_first8(first);
  }
  const unsigned char* data = smem + kGncOffData;
  float tn = 0.0f, tr = 0.0f;
  RefSums ts;
  if (ok) {
    for (int v0 = threadIdx.x; v0 < nvec; v0 += NT * kGnBatch) {
      uint4 v[kGnBatch];
#pragma unroll
      for (int b = 0; b < kGnBatch; ++b) {
        const int k = v0 + b * NT;
        v[b] = k < nvec ? *reinterpret_cast<const uint4*>(data + k * 16) : make_uint4(0, 0, 0, 0);
      }
      float2 f[4];
      Elem<T>::unpack(v[0], f);
      const float kb = f[0].x;
      const float2 nk = make_float2(-kb, -kb);
      float2 a1 = make_float2(0.0f, 0.0f), a2 = make_float2(0.0f, 0.0f);
      float nb = 0.0f;
#pragma unroll
      for (int b = 0; b < kGnBatch; ++b) {
        if (v0 + b * NT < nvec) {
          float2 X[4];
          Elem<T>::unpack(v[b], X);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 d = __fadd2_rn(X[j], nk);
            a1 = __fadd2_rn(a1, d);
            a2 = __ffma2_rn(d, d, a2);
          }
          nb = __fadd_rn(nb, 8.0f);
        }
      }
      const Moments bp = moments_of(nb, __fsub_rn(kb, K), __fadd_rn(a1.x, a1.y), __fadd_rn(a2.x, a2.y));
      if (tn == 0.0f) tr = bp.u;
      ts.add(bp, tr);
      tn = __fadd_rn(tn, nb);
    }
  }
  const Moments mine = tn == 0.0f ? Moments{0.0f, 0.0f, 0.0f} : merged(tn, tr, ts);
  const Moments pm = part_moments<NT>(mine, ok ? nvec : 0, red);
  if (threadIdx.x == 0) {
    part[0] = pm.u;
    part[1] = pm.m;
    *bad = ok ? 0 : 1;
  }

  // (A) every part's statistics are in its CTA's shared memory
  cluster_arrive();
  cluster_wait();

  // warp 0: lane r reads part r over distributed shared memory; the parts
  // are merged around part 0's mean by an xor tree, the same in every CTA
  if (warp == 0) {
    Moments v{0.0f, 0.0f, 0.0f};
    bool b = false;
    if (static_cast<unsigned>(lane) < csize) {
      v.n = static_cast<float>(part_elems(lane, p.part_len, L));
      v.u = __uint_as_float(ld_cluster_u32(base + kGncOffPart, lane));
      v.m = __uint_as_float(ld_cluster_u32(base + kGncOffPart + 4, lane));
      b = ld_cluster_u32(base + kGncOffBad, lane) != 0;
    }
    const bool any_bad = __any_sync(0xffffffffu, b);
    const Moments acc = warp_moments(v, static_cast<float>(L));
    if (lane == 0) {
      const float var = __fmul_rn(acc.m, __frcp_rn(static_cast<float>(L)));
      coef[0] = acc.u;
      coef[1] = rsqrtf(__fadd_rn(var, p.eps));
      coef[2] = K;
      coef[3] = any_bad ? 1.0f : 0.0f;
    }
  }
  // (B) this CTA has read the other CTAs' statistics; it waits for the
  // others' arrival only before it exits
  cluster_arrive();
  __syncthreads();

  if (coef[3] == 0.0f) {
    const float m1 = coef[0], rstd = coef[1];
    const float2 nk = make_float2(-coef[2], -coef[2]);
    const int ch0 = static_cast<int>(span % p.groups) * p.group_channels;
    char* obase = p.out + (span * L + lo) * 2;
    // checked builds: the part's output inside out, else it is not written
    const bool out_ok = in_span(obase, bytes, p.sp_out, p.status);
    const unsigned hw = static_cast<unsigned>(p.hw);
    unsigned ch_end = 0;
    float2 A = make_float2(0.0f, 0.0f), B = make_float2(0.0f, 0.0f);
    for (int v = threadIdx.x; v < nvec && out_ok; v += NT) {
      const unsigned e = static_cast<unsigned>(lo) + static_cast<unsigned>(v) * 8u;   // < L < 2^31
      if (e >= ch_end) {
        const unsigned cl = e / hw;
        ch_end = (cl + 1u) * hw;
        const float* gp = p.gamma + ch0 + cl;
        const float* bq = p.beta + ch0 + cl;
        const bool gb = in_span(gp, 4, p.sp_gamma, p.status) && in_span(bq, 4, p.sp_beta, p.status);
        fold_channel(gb ? __ldg(gp) : 0.0f, gb ? __ldg(bq) : 0.0f, m1, rstd, A, B);
      }
      const uint4 raw = *reinterpret_cast<const uint4*>(data + v * 16);
      store16(obase + static_cast<long long>(v) * 16, silu_affine<T>(raw, nk, A, B));
    }
  }

  // no CTA of the cluster reads this one's shared memory any more
  cluster_wait();
  // copies that did not land in time may still be in flight: wait for them
  // (bounded) before this CTA's shared memory is released
  if (threadIdx.x == 0 && *issued && !ok) {
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(full, 0) && global_timer_ns() - t0 < p.wait_limit_ns) {
    }
  }
}

}  // namespace qknr
