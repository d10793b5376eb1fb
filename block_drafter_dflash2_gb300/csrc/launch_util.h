// Host-side launch helpers shared by the kernel translation units.
#pragma once

#include <cuda_runtime.h>

namespace df {

// Raises `func`'s dynamic shared-memory limit to the device's opt-in maximum (less the
// kernel's static shared memory) once per device, so later launches of any size up to it
// need no attribute call. `done` is the caller's per-device flag array.
inline cudaError_t smem_opt_in(const void* func, unsigned char (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  int optin = 0;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, func)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - (int)fa.sharedSizeBytes)) != cudaSuccess)
    return e;
  if (dev >= 0 && dev < 64) done[dev] = 1;
  return cudaSuccess;
}

}  // namespace df
