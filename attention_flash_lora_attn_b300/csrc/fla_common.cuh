// Shared device helpers of the Flash-LoRA-Attention library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace fla {

// Device error word of this library image.  A kernel whose bounded wait runs
// out stores a nonzero code here (first writer wins) and returns early.
__device__ uint32_t g_device_error;

enum DeviceErrorCode : uint32_t {
  kErrNone = 0,
  kErrDecodeFullWait = 0x101,   // decode consumer: stage never filled
  kErrDecodeEmptyWait = 0x102,  // decode producer: stage never released
  kErrDecodeT5Wait = 0x103,     // tcgen05 decode: any pipeline wait
  kErrBuildFullWait = 0x201,    // LR build MMA warp: operands never landed
  kErrBuildEmptyWait = 0x202,   // LR build producer: stage never released
  kErrBuildAccWait = 0x203,     // LR build epilogue: accumulator never committed
  kErrBuildClusterWait = 0x204, // LR build split-K: a peer CTA never published its partial / finished reading
  kErrPrefillWait = 0x301,      // prefill: any pipeline wait
  kErrSelfTestWait = 0x401,     // fla_selftest_bounded_wait: the wait it was asked to let run out
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

// ---------------------------------------------------------------------------
// Host-side caches of per-device facts, so a launch does no redundant driver
// calls: the SM count and each kernel's raised dynamic shared-memory limit.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

inline int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  return dev;
}

inline int device_sm_count() {
  static std::atomic<int> cache[kMaxDevices];  // 0 = not looked up yet
  const int dev = current_device();
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  n = 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device,
// size): later launches of the same kernel with no more shared memory skip it.
inline cudaError_t ensure_dynamic_smem(const void *kernel, int bytes) {
  struct Entry {
    const void *fn;
    int dev, bytes;
  };
  static std::mutex mu;
  static Entry entries[256];
  static int n_entries = 0;
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_entries; ++i)
    if (entries[i].fn == kernel && entries[i].dev == dev && entries[i].bytes >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n_entries; ++i)
    if (entries[i].fn == kernel && entries[i].dev == dev) {
      entries[i].bytes = bytes;
      return cudaSuccess;
    }
  if (n_entries < 256) entries[n_entries++] = Entry{kernel, dev, bytes};
  return cudaSuccess;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace fla
