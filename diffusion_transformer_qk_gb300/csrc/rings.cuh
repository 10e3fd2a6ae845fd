// The producer side of the AdaLN kernel's row-group stage rings.  The
// consumer warps of a CTA form groups; each group drains its own ring of S
// stages strictly in order.  The producer hands each of the
// CTA's rows to whichever group has a free stage first (searching from the
// group after the last one served), writes the row's index beside the
// stage, and when the rows run out gives every group one stage carrying the
// end mark (-1).  A group that works faster takes more rows.
#pragma once

#include "qknr_ptx.cuh"

namespace qknr {

constexpr int kRingMaxGroups = 16;

// Shared memory of the producer's bookkeeping: per group its next slot, the
// slot's phase and the rows it was given (-1 - rows once it has its mark).
constexpr int kRingPosBytes = 3 * kRingMaxGroups * 4;

struct GroupRings {
  int* pos;
  int n_groups, S;
  uint32_t empty0;     // empty barrier of slot s of group g: empty0 + 8 * (g * S + s)
  int next = 0;

  __device__ __forceinline__ GroupRings(unsigned char* pos_smem, int n_groups_, int S_, uint32_t empty0_)
      : pos(reinterpret_cast<int*>(pos_smem)), n_groups(n_groups_), S(S_), empty0(empty0_) {}

  // one thread, before any use (the producer's own state)
  __device__ __forceinline__ void init() {
    for (int i = 0; i < 3 * kRingMaxGroups; ++i) pos[i] = 0;
  }
  __device__ __forceinline__ int slot(int g) const { return pos[g]; }
  __device__ __forceinline__ bool marked(int g) const { return pos[2 * kRingMaxGroups + g] < 0; }
  __device__ __forceinline__ int given(int g) const {
    const int v = pos[2 * kRingMaxGroups + g];
    return v < 0 ? -1 - v : v;
  }

  // A group without its end mark whose next stage is free, searching from
  // `next`; -1 when the CTA has given up or the wait ran out (then the abort
  // flag and the caller's status word are set).  Between rounds the thread
  // sleeps in the barrier of the first candidate (so with one group it
  // wakes as soon as that stage frees, as a plain wait would) for at most
  // half a microsecond.
  __device__ __forceinline__ int free_group(unsigned long long limit_ns, volatile int* abort_flag, int* status) {
    unsigned long long t0 = 0;
    for (;;) {
      int first = -1;
      for (int i = 0; i < n_groups; ++i) {
        int g = next + i;
        if (g >= n_groups) g -= n_groups;
        if (marked(g)) continue;
        if (first < 0) first = g;
        if (mbar_try_wait(empty0 + 8 * (g * S + pos[g]), static_cast<uint32_t>(pos[kRingMaxGroups + g]) ^ 1u))
          return g;
      }
      if (first < 0 || *abort_flag) return -1;
      if (t0 == 0) t0 = global_timer_ns();
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (status) atomicCAS(status, 0, kStatusTimeout);
        return -1;
      }
      if (mbar_try_wait_sleep(empty0 + 8 * (first * S + pos[first]),
                              static_cast<uint32_t>(pos[kRingMaxGroups + first]) ^ 1u, 500u))
        return first;
    }
  }

  // group g's next stage has been given a row
  __device__ __forceinline__ void advance(int g) {
    if (++pos[g] == S) {
      pos[g] = 0;
      pos[kRingMaxGroups + g] ^= 1;
    }
    ++pos[2 * kRingMaxGroups + g];
    next = g + 1 == n_groups ? 0 : g + 1;
  }

  // group g's next stage has been given the end mark
  __device__ __forceinline__ void mark(int g) {
    pos[2 * kRingMaxGroups + g] = -1 - pos[2 * kRingMaxGroups + g];
    next = g + 1 == n_groups ? 0 : g + 1;
  }

  // Wait (bounded) for the copies of every group's latest S stages, before
  // a CTA that gives up releases its shared memory.
  __device__ __forceinline__ void drain(uint32_t full0, unsigned long long limit_ns) const {
    for (int g = 0; g < n_groups; ++g) {
      const int rows = given(g);
      for (int back = 1; back <= S && back <= rows; ++back) {
        const int j = rows - back;                   // the group's j-th row: slot j % S, phase (j / S) & 1
        const uint32_t bar = full0 + 8 * (g * S + j % S);
        const uint32_t phase = static_cast<uint32_t>((j / S) & 1);
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(bar, phase) && global_timer_ns() - t0 < limit_ns) {
        }
      }
    }
  }
};

}  // namespace qknr
