// Kernel instances for fp16 activations with f32 cos/sin tables.
#include "qknr_internal.h"

namespace qknr {

template <int D>
static const void* pick_fp16_f32(bool rh, bool ex) {
  if (!rh && !ex) return reinterpret_cast<const void*>(&qknr_fused_kernel<__half, float, D, false, false>);
  if (rh && !ex) return reinterpret_cast<const void*>(&qknr_fused_kernel<__half, float, D, true, false>);
  if (!rh && ex) return reinterpret_cast<const void*>(&qknr_fused_kernel<__half, float, D, false, true>);
  return reinterpret_cast<const void*>(&qknr_fused_kernel<__half, float, D, true, true>);
}

const void* kernel_fp16_f32(int D, bool rotate_half, bool expanded) {
  switch (D) {
    case 64: return pick_fp16_f32<64>(rotate_half, expanded);
    case 128: return pick_fp16_f32<128>(rotate_half, expanded);
    default: return nullptr;
  }
}

}  // namespace qknr
