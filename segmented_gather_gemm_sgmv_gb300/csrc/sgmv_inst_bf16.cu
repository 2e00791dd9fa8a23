// sgmv_inst_bf16.cu -- instantiates the shrink / expand / fused kernels for __nv_bfloat16 elements.
#include "sgmv_core.cuh"
#include "sgmv_launch.h"

namespace sgmv {

template <int MODE>
static const void* pick_bf16(int r) {
  switch (r) {
    case 8: return reinterpret_cast<const void*>(&sgmv_kernel<__nv_bfloat16, 8, MODE>);
    case 16: return reinterpret_cast<const void*>(&sgmv_kernel<__nv_bfloat16, 16, MODE>);
    case 32: return reinterpret_cast<const void*>(&sgmv_kernel<__nv_bfloat16, 32, MODE>);
    case 64: return reinterpret_cast<const void*>(&sgmv_kernel<__nv_bfloat16, 64, MODE>);
    default: return nullptr;
  }
}

const void* kernel_bf16(int mode, int r) {
  switch (mode) {
    case kFused: return pick_bf16<kFused>(r);
    case kShrink: return pick_bf16<kShrink>(r);
    case kExpand: return pick_bf16<kExpand>(r);
    default: return nullptr;
  }
}

}  // namespace sgmv
