// Activation quantisation of the dynamic FP8 expert path.
//
// The pages list a compressed-tensors dynamic FP8 checkpoint of the model
// beside the BF16 and NVFP4 ones ("SGLang 原生支持 Reflection 的 Beam 并驱动其
// 生产 API", sections "Highlights" and "BF16, NVFP4 and FP8 Model Support").
// In that scheme the weights are E4M3 with one FP32 scale per output row
// and the activations are quantised per row at run time: a row's scale is
// its largest magnitude over 448 (the largest finite E4M3 value), each
// value is divided by it in FP32 and rounded to the nearest E4M3 value,
// ties to even, saturating at 448.  An all-zero row takes scale 1.  The
// GEMMs (expert_gemm.cu, kind::f8f6f4) multiply the FP32 accumulators by the
// weight row's and the token row's scales.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "launch_once.cuh"
#include "ptx.cuh"

namespace beam {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Two FP32 values -> two E4M3 codes, round to nearest even, saturating
// (the first value in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// One block per row of `cols` BF16 values (cols % 8 == 0, rows 16-byte
// aligned): the row's amax, then its codes and scale.  Rows at or past
// *n_valid (when given) are skipped.  The row is read twice; the second
// read hits the cache.
__global__ void __launch_bounds__(kThreads) quantize_e4m3_rows_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ n_valid, int32_t cols,
    uint8_t* __restrict__ q, float* __restrict__ scale) {
  // programmatic dependent launch: the rows (and n_valid) come from the
  // kernels before this one; once they are visible the next GEMM may start
  // its weight loads
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int64_t row = blockIdx.x;
  if (n_valid && row >= *n_valid) return;
  const uint4* in = reinterpret_cast<const uint4*>(x + row * cols);
  const int n8 = cols / 8;
  float amax = 0.f;
  for (int i = threadIdx.x; i < n8; i += kThreads) {
    const uint4 v = in[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kThreads / 32; ++k) amax = fmaxf(amax, red[k]);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint2* out = reinterpret_cast<uint2*>(q + row * cols);
  for (int i = threadIdx.x; i < n8; i += kThreads) {
    const uint4 v = in[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      c[j] = e4m3x2(__fdiv_rn(bf16_lo(w[j]), s), __fdiv_rn(bf16_hi(w[j]), s));
    out[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
  if (threadIdx.x == 0) scale[row] = s;
}

// The same rule with one warp per row and the row held in registers (V
// 16-byte words per lane: cols <= 256 V): one read of the row, the amax by
// shuffles, no shared memory.  Four rows per 128-thread block.
template <int V>
__global__ void __launch_bounds__(kThreads) quantize_e4m3_rows_warp_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ n_valid, int64_t rows,
    int32_t cols, uint8_t* __restrict__ q, float* __restrict__ scale) {
  ptx::grid_dep_wait();  // as quantize_e4m3_rows_kernel
  ptx::grid_dep_launch();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // row is the same on every lane of the warp: whole warps leave together
  if (row >= rows || (n_valid && row >= *n_valid)) return;
  const uint4* in = reinterpret_cast<const uint4*>(x + row * cols);
  const int n8 = cols / 8;
  uint4 v[V];
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const int i = lane + 32 * j;
    if (i < n8) {
      v[j] = in[i];
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint2* out = reinterpret_cast<uint2*>(q + row * cols);
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const int i = lane + 32 * j;
    if (i < n8) {
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      uint32_t c[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        c[k] = e4m3x2(__fdiv_rn(bf16_lo(w[k]), s), __fdiv_rn(bf16_hi(w[k]), s));
      out[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
  }
  if (lane == 0) scale[row] = s;
}

template <int V>
void launch_warp(const uint16_t* x, const int32_t* n_valid, int64_t rows, int32_t cols,
                 uint8_t* q, float* scale, cudaStream_t s) {
  const int64_t blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
  launch_dependent(quantize_e4m3_rows_warp_kernel<V>, dim3(static_cast<unsigned>(blocks)),
                   dim3(kThreads), 0, s, x, n_valid, rows, cols, q, scale);
}

}  // namespace

void launch_quantize_e4m3_rows(const uint16_t* x, const int32_t* n_valid, int64_t rows,
                               int32_t cols, uint8_t* q, float* scale, cudaStream_t s) {
  if (rows <= 0) return;
  // Many short rows (the h rows of a large batch): one warp per row from
  // registers, 124 -> 102 us on 65536 rows of 2560.  Few rows or long rows
  // (the token rows, decode batches): one block per row, which keeps more
  // loads and divisions in flight per row (5120-wide rows: 28 us against 35
  // with a warp per row; 32 rows: 7 us against 12).
  const int v = (cols / 8 + 31) / 32;  // 16-byte words per lane
  if (rows >= 2048 && v <= 12) {
    if (v <= 4) return launch_warp<4>(x, n_valid, rows, cols, q, scale, s);
    if (v <= 8) return launch_warp<8>(x, n_valid, rows, cols, q, scale, s);
    return launch_warp<12>(x, n_valid, rows, cols, q, scale, s);
  }
  launch_dependent(quantize_e4m3_rows_kernel, dim3(static_cast<unsigned>(rows)), dim3(kThreads), 0,
                   s, x, n_valid, cols, q, scale);
}

}  // namespace beam
