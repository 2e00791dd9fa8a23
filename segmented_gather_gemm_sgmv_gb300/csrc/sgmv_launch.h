// sgmv_launch.h -- host-side glue between the C ABI (sgmv_abi.cu) and the per-dtype kernel
// instantiations (sgmv_inst_*.cu).
#pragma once
#include <cstdint>

namespace sgmv {

// Returns the __global__ function for (mode, rank) of one element type, or nullptr when the
// rank is not instantiated.  mode: 0 fused, 1 shrink, 2 expand.  wide: the long-batch
// instantiation (kThreadsWide threads, one CTA per SM) instead of the default one.
const void* kernel_f32(int mode, int r, bool wide);
const void* kernel_f16(int mode, int r, bool wide);
const void* kernel_bf16(int mode, int r, bool wide);

// The fused kernel over several projections in one launch (lora_apply_multi).
const void* kernel_multi_f32(int r, bool wide);
const void* kernel_multi_f16(int r, bool wide);
const void* kernel_multi_bf16(int r, bool wide);

// The current device's library context for kernels launched outside sgmv_abi.cu: the device
// error word, the SM count and the bounded-wait settings (sgmv_set_wait_limit).
int device_context(int** err, int* sms, uint64_t* wait_ns, int* inject_stall);

}  // namespace sgmv
