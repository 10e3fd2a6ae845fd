// AdaLN kernel instances: activation dtype x modulation dtype x unroll of
// the per-lane chunk loops (1, 2 or 4).
#include "adaln_kernel.cuh"

namespace qknr {

// fp32 modulation doubles the registers a chunk's second pass holds, so its
// instances stop at an unroll of 2 (4 would spill at 17 warps per CTA).
template <typename T, typename MT>
static const void* pick(int unroll) {
  constexpr bool wide = sizeof(MT) == 4;
  switch (unroll) {
    case 1: return reinterpret_cast<const void*>(&adaln_kernel<T, MT, 1>);
    case 2: return reinterpret_cast<const void*>(&adaln_kernel<T, MT, 2>);
    case 4:
      if constexpr (wide)
        return reinterpret_cast<const void*>(&adaln_kernel<T, MT, 2>);
      else
        return reinterpret_cast<const void*>(&adaln_kernel<T, MT, 4>);
    default: return nullptr;
  }
}

// act: 0 bf16, 1 fp16; mod_fp32: scale/shift are fp32 (else the activation
// dtype); unroll: 1, 2 or 4
const void* adaln_kernel_for(int act, bool mod_fp32, int cpl) {
  if (act == 0) return mod_fp32 ? pick<__nv_bfloat16, float>(cpl) : pick<__nv_bfloat16, __nv_bfloat16>(cpl);
  return mod_fp32 ? pick<__half, float>(cpl) : pick<__half, __half>(cpl);
}

}  // namespace qknr
