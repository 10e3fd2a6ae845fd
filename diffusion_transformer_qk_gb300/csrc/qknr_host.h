// Host-side helpers shared by the library's launchers: error text, device
// attribute cache, one-time kernel configuration, address-span checks.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/qknr.h"

namespace qknr_host {

extern thread_local char g_err[512];

// Record a printf-style message for qknr_last_error() and return `s`.
qknr_status fail(qknr_status s, const char* fmt, ...);
qknr_status cuda_fail(cudaError_t e, const char* what);

struct DeviceInfo {
  int num_sms = 0;
  int smem_optin = 0;       // max dynamic shared memory per block (opt-in)
  int smem_per_sm = 0;
  int smem_reserved = 0;    // per-block reservation
  int cooperative = 0;      // cooperative launches supported
};

// Attributes of device `dev`, queried once and cached.
qknr_status device_info(int dev, DeviceInfo* out);

// Set the kernel's dynamic shared memory ceiling to the device maximum
// (once per kernel and device) and return its register count.
qknr_status configure_kernel(const void* fn, int dev, const DeviceInfo& di, int* regs);

// Resident blocks per SM of `fn` at this block size and dynamic shared
// memory on device `dev` (queried once per combination and cached).
qknr_status occupancy(const void* fn, int dev, int block, size_t smem, int* blocks_per_sm);

// Launch `fn` on `stream`; with `overlap`, with programmatic stream
// serialization (the kernel must call griddepcontrol.wait before its first
// global memory access).
qknr_status launch_kernel(const void* fn, int grid, int block, size_t smem, cudaStream_t stream, void** kargs,
                          bool overlap, const char* what);

struct Span {
  uintptr_t lo, hi;   // [lo, hi)
};

// Bytes touched by `rows` rows of `row_bytes` at `stride_bytes` from `base`.
Span span_of(const void* base, long long rows, long long stride_bytes, long long row_bytes);
bool overlaps(Span a, Span b);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace qknr_host
