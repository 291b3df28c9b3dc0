// The dynamic shared-memory opt-in that every kernel of the library needs
// before its first launch on a device.
#pragma once

#include <atomic>

#include <cuda_runtime.h>

namespace fattn {

// Raise ``kern``'s dynamic shared-memory limit to ``smem`` bytes on the
// current device, once per device for the first 64 devices (``done`` is the
// kernel's own flag array, static at the call site).  Setting the attribute
// again is harmless, so threads that race on a device's first launch both
// set it; the atomic flags keep the check itself free of data races.
template <typename Kernel>
cudaError_t smem_opt_in(Kernel kern, int smem, std::atomic<bool> (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire))
    return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64)
    done[dev].store(true, std::memory_order_release);
  return e;
}

}  // namespace fattn
