// Internal interface between the C-ABI launcher and the kernel instances.
#pragma once

#include "qknr_kernel.cuh"

namespace qknr {

// Kernel entry for (activation dtype, table dtype) with head_dim D, pairing
// and table layout, or nullptr when that instance does not exist.
// act: 0 bf16, 1 fp16.  Defined one (act, table) pair per translation unit.
const void* kernel_bf16_f32(int D, bool rotate_half, bool expanded);
const void* kernel_bf16_bf16(int D, bool rotate_half, bool expanded);
const void* kernel_fp16_f32(int D, bool rotate_half, bool expanded);
const void* kernel_fp16_bf16(int D, bool rotate_half, bool expanded);

}  // namespace qknr
