// Host-side launch set-up shared by the kernel launchers.
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <utility>

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

// ------------------------------------------- programmatic dependent launch
// The layer's later kernels (token-row quantisation and gathers, expert
// GEMMs, combine) are launched with programmatic stream serialization
// (SGLang post "SGLang 原生支持 Reflection 的 Beam 并驱动其生产 API", section
// "Fusion Optimizations": a kernel sets up and loads weights before its
// dependency wait).  Such a kernel may start while the kernel before it
// still runs, so each one executes griddepcontrol.wait before it reads
// anything that kernel writes, and writes nothing that kernel reads.  Reads
// before the wait (a GEMM's tile list and weights) are allowed only of data
// written two or more kernels earlier: every kernel here that lets its
// successor start early (griddepcontrol.launch_dependents) does so after its
// own wait, so by then all earlier kernels have completed.  A kernel that
// never triggers lets its successor start when it completes.
constexpr int kProgrammaticLaunch = 1;

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace beam
