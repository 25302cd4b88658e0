// Launchers of the grouped expert GEMMs (device code: expert_gemm_kernel.cuh).
#include "expert_gemm_kernel.cuh"
#include "launch_once.cuh"

namespace beam {
namespace {

template <int NT, int MODE, bool F8>
cudaError_t launch_impl(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                        const GemmArgs& p, int grid, cudaStream_t s) {
  using C = Cfg<NT, MODE>;
  auto kern = expert_gemm_kernel<NT, MODE, F8>;
  const cudaError_t err = smem_limit_once<expert_gemm_kernel<NT, MODE, F8>>(C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(a0, a1, b, p);
  return cudaGetLastError();
}

}  // namespace

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
