// Opting a kernel into more than 48 KB of dynamic shared memory.
//
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) is a setting of the
// current device's context, so a process that calls on device 0 and then on
// device 1 must set it on both.  Each launch site keeps one flag per device
// ordinal (an array of its own: the flag belongs to one kernel instantiation)
// and sets the attribute the first time it launches on a device.  The flags
// are atomics because the C ABI may be called from several host threads;
// setting the attribute twice is harmless.
#pragma once

#include <atomic>

#include <cuda_runtime.h>

namespace attn {

constexpr int kMaxAttrDevices = 64;

using DeviceFlags = std::atomic<bool>[kMaxAttrDevices];

template <typename Kern>
cudaError_t ensure_dyn_smem(Kern kern, int bytes, DeviceFlags& configured) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxAttrDevices;
  if (tracked && configured[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) configured[dev].store(true, std::memory_order_release);
  return e;
}

}  // namespace attn
