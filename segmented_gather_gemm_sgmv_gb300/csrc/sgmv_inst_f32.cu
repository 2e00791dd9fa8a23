// sgmv_inst_f32.cu -- instantiates the shrink / expand / fused kernels for float elements.
#include "sgmv_core.cuh"
#include "sgmv_launch.h"

namespace sgmv {

template <int MODE>
static const void* pick_f32(int r) {
  switch (r) {
    case 8: return reinterpret_cast<const void*>(&sgmv_kernel<float, 8, MODE>);
    case 16: return reinterpret_cast<const void*>(&sgmv_kernel<float, 16, MODE>);
    case 32: return reinterpret_cast<const void*>(&sgmv_kernel<float, 32, MODE>);
    case 64: return reinterpret_cast<const void*>(&sgmv_kernel<float, 64, MODE>);
    default: return nullptr;
  }
}

const void* kernel_f32(int mode, int r) {
  switch (mode) {
    case kFused: return pick_f32<kFused>(r);
    case kShrink: return pick_f32<kShrink>(r);
    case kExpand: return pick_f32<kExpand>(r);
    default: return nullptr;
  }
}

}  // namespace sgmv
