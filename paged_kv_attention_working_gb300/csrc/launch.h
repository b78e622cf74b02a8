// Host-side launch helpers: the per-device dynamic shared memory limit of a
// kernel, and launches with programmatic dependent launch.
//
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
#include <utility>

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

// Launch with programmatic dependent launch: the grid may be scheduled while
// the previous kernel on the stream is still running (once every CTA of that
// kernel has started), so its launch latency and CTA set-up overlap the
// predecessor's tail.  Every kernel launched this way executes
// griddepcontrol.wait (pdl_wait) before it touches global memory; that wait
// returns once the preceding grid has completed and its writes are visible,
// so the stream order holds for every byte the kernel reads or writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pie
