// Interface of the persistent grouped expert GEMM (expert_gemm.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace beam {

constexpr int kModeDown = 0;    // y = w * (h W_d^T), FP32 out
constexpr int kModeGateUp = 1;  // h = bf16(silu(x W_g^T) * (x W_u^T))
constexpr int kModeDownPair = 2;  // as kModeDown over pairs of 128-row W_d blocks
                                  // (m_blocks = d / 256)

struct GemmArgs {
  const int32_t* counts;   // [E] rows per expert
  const int32_t* perm_src; // [rows] permuted row -> token * topk + slot (gate/up gather)
  int32_t topk;
  const int32_t* offsets;  // [E+1] first row of each expert in the token operand
  const float* perm_w;     // [rows] routing weight per row (down)
  uint16_t* h_out;         // gate/up: h [rows, F] BF16
  float* f32_out;          // down: y [rows, d] FP32
  const int32_t* out_rows; // down: output row of each permuted row (nullptr: the same row)
  int32_t out_ld;          // elements per output row
  int32_t E;               // experts in the tile list
  int32_t rows_per_expert; // weight rows of one expert (A operand)
  int32_t m_blocks;        // rows_per_expert / 128
  int32_t k_blocks;        // A's K / 64 (BF16) or / 128 (E4M3): 128-byte K blocks
  int32_t b_k_blocks;      // the token operand's, == k_blocks
  int32_t weight_evict_first;
  uint32_t* status;
  uint64_t wait_limit_ns;
  int32_t withhold_first_load;
  // E4M3 operands only: FP32 scale of every weight row ([E * rows_per_expert];
  // a0's rows, and a1's for gate/up) and of every token operand row: per
  // token for gate/up ([T], looked up through perm_src), per permuted row
  // for down ([rows]).  The accumulators are multiplied by both.
  const float* a0_scale;
  const float* a1_scale;
  const float* b_scale;
  // extents for the debug build's bounds checks: weight rows of the A tensor
  // map (E * rows_per_expert), rows of the token tensor map, rows of the
  // output buffer
  int32_t a_rows;
  int32_t b_rows;
  int32_t out_rows_cap;
};

// Persistent grouped GEMM; `nt` is the token-block width, 16 or 256 (the
// paired down mode takes 256 only).  `f8`: both operands are E4M3 (K blocks of 128 elements)
// instead of BF16 (K blocks of 64); the only other difference is the
// scaling in the epilogue.  Tensor maps are encoded by the caller.
cudaError_t launch_grouped_gemm(int mode, int nt, const CUtensorMap& a0, const CUtensorMap& a1,
                                const CUtensorMap& b, const GemmArgs& a, int grid,
                                cudaStream_t s, bool f8 = false);

// The same GEMMs for 256-token blocks on clusters of two CTAs that share
// M = 256 MMAs (expert_gemm_pair_kernel.cuh): gate/up over 256-row blocks of
// F (m_blocks = d_ff / 256), down over 512-row blocks of d, two 256-row
// accumulators (m_blocks = d / 512).  The token tensor map's box is 128
// rows (each CTA stages half a block).
// At most max_pairs clusters; as many as can be resident.
cudaError_t launch_grouped_gemm_pair(bool gateup, const CUtensorMap& a0, const CUtensorMap& a1,
                                     const CUtensorMap& b, const GemmArgs& a, int max_pairs,
                                     cudaStream_t s, bool f8 = false);

}  // namespace beam
