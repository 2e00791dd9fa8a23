// sgmv_inst_f16.cu -- instantiates the shrink / expand / fused kernels for __half elements.
#include "sgmv_core.cuh"
#include "sgmv_launch.h"

namespace sgmv {

template <int MODE>
static const void* pick_f16(int r, bool wide) {
  switch (r) {
    case 8: return kernel_ptr<__half, 8, MODE>(wide);
    case 16: return kernel_ptr<__half, 16, MODE>(wide);
    case 32: return kernel_ptr<__half, 32, MODE>(wide);
    case 64: return kernel_ptr<__half, 64, MODE>(wide);
    default: return nullptr;
  }
}

const void* kernel_f16(int mode, int r, bool wide) {
  switch (mode) {
    case kFused: return pick_f16<kFused>(r, wide);
    case kShrink: return pick_f16<kShrink>(r, wide);
    case kExpand: return pick_f16<kExpand>(r, wide);
    default: return nullptr;
  }
}

const void* kernel_multi_f16(int r, bool wide) {
  switch (r) {
    case 8: return multi_kernel_ptr<__half, 8>(wide);
    case 16: return multi_kernel_ptr<__half, 16>(wide);
    case 32: return multi_kernel_ptr<__half, 32>(wide);
    case 64: return multi_kernel_ptr<__half, 64>(wide);
    default: return nullptr;
  }
}

}  // namespace sgmv
