// Declarations shared by the host entry points and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace beam {

// Status codes latched by kernels (values of beam_status_t).
constexpr uint32_t kStatusTimeout = 5;
constexpr uint32_t kStatusDeviceCheck = 6;

__device__ __forceinline__ void latch_status(uint32_t* status, uint32_t code) {
  atomicCAS(status, 0u, code);
}

// Bounds checks of the debug build.  Compiled with -DBEAM_DEVICE_CHECKS=1
// (build(checked=True)), every checked index -- a permuted row, a TMA
// coordinate, a TMEM column, a tile -- that falls outside its buffer
// latches BEAM_ERR_DEVICE_CHECK in the call's status word, and the caller
// skips the access (or clamps a copy's coordinates, so that the barrier the
// copy signals still completes).  Nothing traps.  The default build compiles
// the checks out: in_bounds() is then `true`.
#ifndef BEAM_DEVICE_CHECKS
#define BEAM_DEVICE_CHECKS 0
#endif

__device__ __forceinline__ bool in_bounds(bool ok, uint32_t* status) {
#if BEAM_DEVICE_CHECKS
  if (!ok) latch_status(status, kStatusDeviceCheck);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}

// ---------------------------------------------------------------- routing
struct RouterArgs {
  const uint16_t* x;       // [T, d] bf16
  const float* w;          // [E, d]
  float* part;             // [ksplit, T, E]
  int64_t T;
  int32_t d, E;
  int32_t k_chunk;         // K elements per split (multiple of 32)
};

struct SelectArgs {
  const float* part;       // [ksplit, T, E] partial logits (ksplit == 1: logits)
  int32_t ksplit;
  const float* bias;       // [E]
  int64_t T;
  int32_t E, G, kg, k;
  float alpha;
  int32_t* idx;            // [T, k]
  float* w;                // [T, k]
  float* logits;           // [T, E] or nullptr (written when ksplit > 1 or copy wanted)
};

struct PermuteArgs {
  const int32_t* idx;      // [TK]
  const float* w;          // [TK]
  int64_t TK;
  int32_t E;
  int32_t* counts;         // [E]
  int32_t* offsets;        // [E+1]
  int32_t* perm_src;       // [TK]
  int32_t* pair_row;       // [TK]
  float* perm_w;           // [TK]
  uint32_t* status;
  int32_t id_base;         // idx holds expert ids id_base .. id_base + E - 1
};

void launch_router(const RouterArgs& a, int ksplit, cudaStream_t s);
void launch_select(const SelectArgs& a, cudaStream_t s);
void launch_permute(const PermuteArgs& a, cudaStream_t s);
// the same permutation as a counting sort in one cooperative launch (large
// batches); hist: int32 [ceil(TK / 1024), E] scratch
cudaError_t launch_permute_sort(const PermuteArgs& a, int32_t* hist, int num_sms, cudaStream_t s);
constexpr int64_t kPermuteSortChunk = 1024;
// expert-parallel dispatch metadata: per packed row its expert and weight,
// and the rows bound for each of n_ranks owners
void launch_ep_pack(const int32_t* idx, const int32_t* perm_src, const float* perm_w,
                    const int32_t* offsets, int64_t TK, int32_t E, int32_t n_ranks,
                    int32_t* send_expert, float* send_w, int32_t* send_counts, cudaStream_t s);
// router partials + selection + permutation in one cooperative launch
cudaError_t launch_fused_route(const RouterArgs& ra, int ksplit, const SelectArgs& sa,
                               const PermuteArgs& pa, int num_sms, cudaStream_t s);
void launch_gather(const uint16_t* x, const int32_t* perm_src, const int32_t* n_valid, int64_t TK,
                   int32_t k, int32_t d, uint16_t* x_perm, cudaStream_t s);
// token rows x [T, n16 16-bit words] -> each token's k permuted rows
// pair_row[t * k + j] of x_perm (each row read once; k <= 32).  `status`
// receives the debug build's bounds-check failures.
void launch_scatter_tokens(const uint16_t* x, const int32_t* pair_row, int64_t T, int32_t k,
                           int32_t n16, uint16_t* x_perm, uint32_t* status, cudaStream_t s);
void launch_combine(const float* y, const int32_t* pair_row, int64_t T, int32_t k, int32_t d,
                    uint16_t* out, uint32_t* status, cudaStream_t s);

// the decoder's sublayer boundary after the layer: post-norm, depth-scaled
// residual add, next pre-norm
struct BoundaryArgs {
  const uint16_t* g_post;  // [d] BF16 RMSNorm weight of the layer's output
  const uint16_t* g_pre;   // [d] BF16 RMSNorm weight of the next sublayer's input
  uint16_t* residual;      // [T, d] BF16 residual stream, read and overwritten
  uint16_t* next_x;        // [T, d] BF16 next sublayer's input
  float eps;
  float c_h, c_x;          // sqrt((n-1)/n), 1/sqrt(n) for the n-th residual add
};
// combine (as launch_combine, into out) fused with the boundary; d*4 bytes of
// shared memory per block
cudaError_t launch_combine_boundary(const float* y, const int32_t* pair_row, int64_t T, int32_t k,
                                    int32_t d, uint16_t* out, const BoundaryArgs& b,
                                    uint32_t* status, cudaStream_t s);

// W_r [E, d] FP32 -> planes [E, 3d] BF16 (hi | mid | lo, W = hi + mid + lo to
// within 2^-24 relative).
void launch_router_split(const float* w, int32_t E, int32_t d, uint16_t* planes, cudaStream_t s);

// logits [T, E] = x [T, d] (BF16) * planes^T on the tensor cores, K-groups
// summed in FP32 (E % 128 == 0, d % 128 == 0).  With ksplit > 1, split c of
// the K ranges writes its partial logits to logits + c * T * E (the caller
// adds the ksplit partials in order).
cudaError_t launch_router_tc(const CUtensorMap& w_planes, const CUtensorMap& x, float* logits,
                             int64_t T, int32_t E, int32_t d, int32_t ksplit, uint32_t* status,
                             uint64_t wait_limit_ns, int num_sms, cudaStream_t s);
// The K split launch_router_tc uses for T tokens on num_sms SMs (>= 1).
int router_tc_ksplit(int64_t T, int32_t E, int32_t d, int num_sms);

// ------------------------------------------------------- NVFP4 and MXFP8
// Arguments of the block-scaled grouped GEMMs (NVFP4, or MXFP8 where noted).
struct Fp4GemmArgs {
  const int32_t* counts;
  const int32_t* offsets;
  const float* perm_w;     // [rows] routing weight (down)
  const uint8_t* sfa0;     // blocked E4M3 (MXFP8: E8M0) weight scales (gate or down)
  const uint8_t* sfa1;     // blocked weight scales (up)
  const float* gs0;        // [E] FP32 scale (gate or down); unused for MXFP8
  const float* gs1;        // [E] FP32 scale (up); unused for MXFP8
  uint8_t* hq;             // gate/up out: h codes [rows, F/2] (MXFP8: [rows, F])
  uint8_t* hsf;            // gate/up out: h scales [rows, F/4], a 16-byte slot per 64
                           // (MXFP8: [rows, F/8], a 16-byte slot per 128)
  float* y;                // down out: [rows, d]
  const int32_t* out_rows; // down: output row of each permuted row (nullptr: the same row)
  int32_t out_ld;          // F (gate/up) or d (down), in elements
  int32_t E;
  int32_t rows_per_expert;
  int32_t m_blocks;
  int32_t k_blocks;        // K / 256 (MXFP8: K / 128)
  int32_t weight_evict_first;
  uint32_t* status;
  uint64_t wait_limit_ns;
  // extents for the debug build's bounds checks: weight rows (E * N), token
  // operand rows, output rows
  int32_t a_rows;
  int32_t b_rows;
  int32_t out_rows_cap;
};

// ---------------------------------------------------------------- W4A16
struct W4a16GemmArgs {
  const int32_t* counts;
  const int32_t* offsets;
  const float* perm_w;     // [rows] routing weight (down)
  const uint8_t* sfa0;     // blocked E4M3 weight scales (gate or down)
  const uint8_t* sfa1;     // blocked E4M3 weight scales (up)
  const float* gs0;        // [E] FP32 scale (gate or down)
  const float* gs1;        // [E] FP32 scale (up)
  uint16_t* h_out;         // gate/up out: h [rows, F] F16
  float* y_out;            // down out: [rows, d] FP32
  int32_t out_ld;          // elements per output row
  int32_t E;
  int32_t rows_per_expert;
  int32_t m_blocks;
  int32_t k_blocks;        // K / 256
  int32_t weight_evict_first;
  uint32_t* status;
  uint64_t wait_limit_ns;
  // extents for the debug build's bounds checks (as Fp4GemmArgs)
  int32_t a_rows;
  int32_t b_rows;
  int32_t out_rows_cap;
};
// permuted token rows -> F16 [rows, d] (saturating at 65504)
void launch_gather_f16(const uint16_t* x, const int32_t* perm_src, const int32_t* n_valid,
                       int64_t TK, int32_t k, int32_t d, uint16_t* x16, cudaStream_t s);
// NVFP4 weights x F16 activations grouped GEMM, nt = 16 | 32; b maps F16 rows
// (box 64 x nt, 128-byte swizzle); the down GEMM works on pairs of adjacent
// 128-row weight blocks (m_blocks = d / 256)
cudaError_t launch_w4a16_gemm(bool gateup, int nt, const CUtensorMap& a0, const CUtensorMap& a1,
                              const CUtensorMap& b, const W4a16GemmArgs& p, int grid,
                              cudaStream_t s);

// [rows, S] row-major E4M3 scales -> 128-row x 4-scale blocks (see nvfp4.cu)
void launch_pack_scales(const uint8_t* src, int64_t rows, int64_t S, uint8_t* dst, cudaStream_t s);
// BF16 rows [rows, cols] -> E4M3 codes [rows, cols] and one FP32 scale per
// row (amax / 448); rows at or past *n_valid, when given, are skipped
void launch_quantize_e4m3_rows(const uint16_t* x, const int32_t* n_valid, int64_t rows,
                               int32_t cols, uint8_t* q, float* scale, cudaStream_t s);
// token rows x [T, d] -> NVFP4 codes [rows, d/2] and scales [rows, d/4] (one
// 16-byte slot, 4 scales + padding, per 64 elements) of each token's k
// permuted rows pair_row[t * k + j]; each token is quantised once (k <= 32)
void launch_quantize_tokens(const uint16_t* x, const int32_t* pair_row, int64_t T, int32_t k,
                            int32_t d, uint8_t* xq, uint8_t* xsf, uint32_t* status,
                            cudaStream_t s);
// block-scaled FP4 grouped GEMM, nt = 16 | 32; sfb maps the token scales; the
// down GEMM works on pairs of adjacent 128-row weight blocks (m_blocks = d / 256)
cudaError_t launch_fp4_gemm(bool gateup, int nt, const CUtensorMap& a0, const CUtensorMap& a1,
                            const CUtensorMap& b, const CUtensorMap& sfb, const Fp4GemmArgs& p,
                            int grid, cudaStream_t s);
// token rows x [T, d] -> MX codes [rows, d] and E8M0 scales [rows, d/8] (one
// 16-byte slot, 4 scales + padding, per 128 elements) of each token's k
// permuted rows pair_row[t * k + j] (k <= 32)
void launch_quantize_tokens_mx(const uint16_t* x, const int32_t* pair_row, int64_t T, int32_t k,
                               int32_t d, uint8_t* xq, uint8_t* xsf, uint32_t* status,
                               cudaStream_t s);
// the MXFP8 grouped GEMM (E4M3 x E4M3, E8M0 per 32), as launch_fp4_gemm
cudaError_t launch_mxfp8_gemm(bool gateup, int nt, const CUtensorMap& a0, const CUtensorMap& a1,
                              const CUtensorMap& b, const CUtensorMap& sfb, const Fp4GemmArgs& p,
                              int grid, cudaStream_t s);

}  // namespace beam
