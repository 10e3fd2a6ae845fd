// Kernel instances for fp16 activations with bf16 cos/sin tables.
#include "qknr_internal.h"

namespace qknr {

template <int D>
static const void* pick_fp16_bf16(bool rh, bool ex) {
  if (!rh && !ex) return reinterpret_cast<const void*>(&qknr_fused_kernel<__half, __nv_bfloat16, D, false, false>);
  if (rh && !ex) return reinterpret_cast<const void*>(&qknr_fused_kernel<__half, __nv_bfloat16, D, true, false>);
  if (!rh && ex) return reinterpret_cast<const void*>(&qknr_fused_kernel<__half, __nv_bfloat16, D, false, true>);
  return reinterpret_cast<const void*>(&qknr_fused_kernel<__half, __nv_bfloat16, D, true, true>);
}

const void* kernel_fp16_bf16(int D, bool rotate_half, bool expanded) {
  switch (D) {
    case 64: return pick_fp16_bf16<64>(rotate_half, expanded);
    case 128: return pick_fp16_bf16<128>(rotate_half, expanded);
    default: return nullptr;
  }
}

}  // namespace qknr
