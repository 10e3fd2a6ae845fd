// AdaLN kernel instances: activation dtype x modulation dtype x chunks per lane.
#include "adaln_kernel.cuh"

namespace qknr {

template <typename T, typename MT>
static const void* pick(int cpl) {
  switch (cpl) {
    case 1: return reinterpret_cast<const void*>(&adaln_kernel<T, MT, 1>);
    case 2: return reinterpret_cast<const void*>(&adaln_kernel<T, MT, 2>);
    case 3: return reinterpret_cast<const void*>(&adaln_kernel<T, MT, 3>);
    default: return nullptr;
  }
}

// act: 0 bf16, 1 fp16; mod_fp32: scale/shift are fp32 (else the activation dtype)
const void* adaln_kernel_for(int act, bool mod_fp32, int cpl) {
  if (act == 0) return mod_fp32 ? pick<__nv_bfloat16, float>(cpl) : pick<__nv_bfloat16, __nv_bfloat16>(cpl);
  return mod_fp32 ? pick<__half, float>(cpl) : pick<__half, __half>(cpl);
}

}  // namespace qknr
