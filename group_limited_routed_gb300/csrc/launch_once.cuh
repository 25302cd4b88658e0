// Host-side launch set-up shared by the kernel launchers.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace beam {

// ------------------------------------------------- per-device launch set-up
// Kernel attributes and occupancy belong to each device's copy of a kernel.
// These helpers do the host-side work once per device and kernel, so later
// calls launch without it (and can be captured into a CUDA graph).
constexpr int kMaxDevices = 64;

// Raises Kern's dynamic shared-memory limit to `bytes` on the current device.
template <auto Kern>
cudaError_t smem_limit_once(int bytes) {
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

// Resident blocks of Kern per SM on the current device (threads per block,
// no dynamic shared memory); 0 when the query fails.
template <auto Kern>
int blocks_per_sm_once(int threads) {
  static std::mutex mu;
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, Kern, threads, 0) != cudaSuccess) return 0;
    cached[dev] = v;
  }
  return cached[dev];
}

}  // namespace beam
