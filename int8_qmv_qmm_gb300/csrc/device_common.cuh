// Device-side helpers shared by the libqlin kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qlin {

// 16-bit storage types of activations, scales and biases.
template <typename T>
struct Act;

template <>
struct Act<__half> {
  using T2 = __half2;
  static __device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
  static __device__ __forceinline__ __half from_f32_rn(float v) { return __float2half_rn(v); }
  // 0x6400 is 1024.0 in binary16: OR-ing a code q < 1024 into the low mantissa
  // bits gives exactly 1024 + q.
  static constexpr uint32_t kMagic2 = 0x64006400u;
  static constexpr float kMagicValue = 1024.0f;
};

template <>
struct Act<__nv_bfloat16> {
  using T2 = __nv_bfloat162;
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32_rn(float v) {
    return __float2bfloat16_rn(v);
  }
  // 0x4300 is 128.0 in bfloat16: OR-ing a code q < 128 gives exactly 128 + q.
  static constexpr uint32_t kMagic2 = 0x43004300u;
  static constexpr float kMagicValue = 128.0f;
};

__device__ __forceinline__ float u32_as_f32(uint32_t v) { return __uint_as_float(v); }

// Programmatic dependent launch: wait until the preceding kernel on the stream
// has completed and its writes are visible (returns at once when the launch
// has no programmatic dependency), and allow the next kernel to launch early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace qlin
