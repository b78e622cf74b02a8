// Per-device set-up of a kernel's dynamic shared memory limit.
//
// cudaFuncAttributeMaxDynamicSharedMemorySize belongs to the current
// device's context, so a kernel that needs more than 48 KB must have it set
// once on every device it runs on.  Each kernel instantiation keeps one flag
// per device ordinal; the flags are atomics, so host threads that launch on
// different devices (or race on the same one) stay correct -- at worst two
// threads both set the attribute, which is harmless.
#pragma once
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

namespace pie {

constexpr int kMaxDeviceOrdinals = 256;

template <auto Kernel>
cudaError_t ensure_smem_attr(int bytes) {
  static std::atomic<uint8_t> done[kMaxDeviceOrdinals];  // zero-initialised
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDeviceOrdinals;
  if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) done[dev].store(1, std::memory_order_release);
  return e;
}

}  // namespace pie
