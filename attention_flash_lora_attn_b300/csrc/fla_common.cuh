// Shared device helpers of the Flash-LoRA-Attention library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fla {

// Device error word of this library image.  A kernel whose bounded wait runs
// out stores a nonzero code here (first writer wins) and returns early.
__device__ uint32_t g_device_error;

enum DeviceErrorCode : uint32_t {
  kErrNone = 0,
  kErrDecodeFullWait = 0x101,   // decode consumer: stage never filled
  kErrDecodeEmptyWait = 0x102,  // decode producer: stage never released
  kErrBuildFullWait = 0x201,    // LR build MMA warp: operands never landed
  kErrBuildEmptyWait = 0x202,   // LR build producer: stage never released
  kErrBuildAccWait = 0x203,     // LR build epilogue: accumulator never committed
  kErrPrefillWait = 0x301,      // prefill: any pipeline wait
};

__device__ __forceinline__ void set_device_error(uint32_t code) {
  atomicCAS(&g_device_error, 0u, code);
}

// Wall-clock bound for every spin-wait in the library (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace fla
