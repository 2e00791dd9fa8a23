// sgmv_inst_bf16.cu -- instantiates the shrink / expand / fused kernels for __nv_bfloat16 elements.
#include "sgmv_core.cuh"
#include "sgmv_launch.h"

namespace sgmv {

template <int MODE>
static const void* pick_bf16(int r, bool wide) {
  switch (r) {
    case 8: return kernel_ptr<__nv_bfloat16, 8, MODE>(wide);
    case 16: return kernel_ptr<__nv_bfloat16, 16, MODE>(wide);
    case 32: return kernel_ptr<__nv_bfloat16, 32, MODE>(wide);
    case 64: return kernel_ptr<__nv_bfloat16, 64, MODE>(wide);
    default: return nullptr;
  }
}

const void* kernel_bf16(int mode, int r, bool wide) {
  switch (mode) {
    case kFused: return pick_bf16<kFused>(r, wide);
    case kShrink: return pick_bf16<kShrink>(r, wide);
    case kExpand: return pick_bf16<kExpand>(r, wide);
    default: return nullptr;
  }
}

const void* kernel_multi_bf16(int r, bool wide) {
  switch (r) {
    case 8: return multi_kernel_ptr<__nv_bfloat16, 8>(wide);
    case 16: return multi_kernel_ptr<__nv_bfloat16, 16>(wide);
    case 32: return multi_kernel_ptr<__nv_bfloat16, 32>(wide);
    case 64: return multi_kernel_ptr<__nv_bfloat16, 64>(wide);
    default: return nullptr;
  }
}

}  // namespace sgmv
