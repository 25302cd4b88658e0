// Launchers of the grouped expert GEMMs (device code: expert_gemm_kernel.cuh,
// expert_gemm_pair_kernel.cuh).
#include <algorithm>
#include <mutex>

#include "expert_gemm_kernel.cuh"
#include "expert_gemm_pair_kernel.cuh"
#include "launch_once.cuh"

namespace beam {
namespace {

// The clusters of two CTAs that can be resident at once on the current
// device (queried once per device and kernel; 0 if the query fails).
template <auto Kern>
int pair_clusters_once(const cudaLaunchConfig_t& cfg) {
  static std::mutex mu;
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, Kern, &cfg) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int MODE, bool F8>
cudaError_t launch_pair_impl(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                             const GemmArgs& p, int max_pairs, cudaStream_t s) {
  using C = PairCfg<MODE>;
  const cudaError_t err =
      smem_limit_once<expert_gemm_pair_kernel<MODE, F8>>(static_cast<int>(C::SMEM_BYTES));
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
  cfg.gridDim = dim3(2);
  // a persistent grid of as many pairs as can be resident (whole waves)
  const int resident = pair_clusters_once<expert_gemm_pair_kernel<MODE, F8>>(cfg);
  if (resident <= 0) return cudaErrorUnknown;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * std::max(1, std::min(resident, max_pairs))));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, expert_gemm_pair_kernel<MODE, F8>, a0, a1, b, p);
}

template <int NT, int MODE, bool F8>
cudaError_t launch_impl(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                        const GemmArgs& p, int grid, cudaStream_t s) {
  using C = Cfg<NT, MODE>;
  const cudaError_t err = smem_limit_once<expert_gemm_kernel<NT, MODE, F8>>(C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  return launch_dependent(expert_gemm_kernel<NT, MODE, F8>, dim3(grid), dim3(C::THREADS),
                          C::SMEM_BYTES, s, a0, a1, b, p);
}

}  // namespace

cudaError_t launch_grouped_gemm_pair(bool gateup, const CUtensorMap& a0, const CUtensorMap& a1,
                                     const CUtensorMap& b, const GemmArgs& a, int max_pairs,
                                     cudaStream_t s, bool f8) {
  if (gateup)
    return f8 ? launch_pair_impl<kModeGateUp, true>(a0, a1, b, a, max_pairs, s)
              : launch_pair_impl<kModeGateUp, false>(a0, a1, b, a, max_pairs, s);
  return f8 ? launch_pair_impl<kModeDownPair, true>(a0, a0, b, a, max_pairs, s)
            : launch_pair_impl<kModeDownPair, false>(a0, a0, b, a, max_pairs, s);
}

cudaError_t launch_grouped_gemm(int mode, int nt, const CUtensorMap& a0, const CUtensorMap& a1,
                                const CUtensorMap& b, const GemmArgs& a, int grid,
                                cudaStream_t s, bool f8) {
  if (f8) {
    switch (mode) {
      case kModeGateUp:
        if (nt == 16) return launch_impl<16, kModeGateUp, true>(a0, a1, b, a, grid, s);
        if (nt == 256) return launch_impl<256, kModeGateUp, true>(a0, a1, b, a, grid, s);
        break;
      case kModeDown:
        if (nt == 16) return launch_impl<16, kModeDown, true>(a0, a0, b, a, grid, s);
        if (nt == 256) return launch_impl<256, kModeDown, true>(a0, a0, b, a, grid, s);
        break;
      case kModeDownPair:
        if (nt == 256) return launch_impl<256, kModeDownPair, true>(a0, a0, b, a, grid, s);
        break;
    }
    return cudaErrorInvalidValue;
  }
  switch (mode) {
    case kModeGateUp:
      if (nt == 16) return launch_impl<16, kModeGateUp, false>(a0, a1, b, a, grid, s);
      if (nt == 256) return launch_impl<256, kModeGateUp, false>(a0, a1, b, a, grid, s);
      break;
    case kModeDown:
      if (nt == 16) return launch_impl<16, kModeDown, false>(a0, a0, b, a, grid, s);
      if (nt == 256) return launch_impl<256, kModeDown, false>(a0, a0, b, a, grid, s);
      break;
    case kModeDownPair:
      if (nt == 256) return launch_impl<256, kModeDownPair, false>(a0, a0, b, a, grid, s);
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace beam
