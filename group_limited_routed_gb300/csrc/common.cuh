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
};

void launch_router(const RouterArgs& a, int ksplit, cudaStream_t s);
void launch_select(const SelectArgs& a, cudaStream_t s);
void launch_permute(const PermuteArgs& a, cudaStream_t s);
void launch_gather(const uint16_t* x, const int32_t* perm_src, const int32_t* n_valid, int64_t TK,
                   int32_t k, int32_t d, uint16_t* x_perm, cudaStream_t s);
void launch_combine(const float* y, const int32_t* pair_row, int64_t T, int32_t k, int32_t d,
                    uint16_t* out, cudaStream_t s);

// ---------------------------------------------------------------- expert GEMMs
struct GemmArgs {
  const int32_t* counts;   // [E]
  const int32_t* offsets;  // [E+1]
  const float* perm_w;     // [TK] (down GEMM epilogue)
  uint16_t* h_out;         // gate/up: h [TK, F] BF16
  float* y_out;            // down: y [TK, d] FP32
  int32_t out_ld;          // elements per output row
  int32_t E;
  int32_t rows_per_expert; // weight rows of one expert (F or d)
  int32_t m_blocks;        // rows_per_expert / 128
  int32_t k_blocks;        // K / 64
  uint32_t* status;
  uint64_t wait_limit_ns;
  int32_t withhold_first_load;
};

// Host-side launch of the grouped expert GEMMs; tensor maps are encoded by
// the caller.  `nt` selects the token-tile width (16 or 128).
cudaError_t launch_gateup(const CUtensorMap& wg, const CUtensorMap& wu, const CUtensorMap& xp,
                          const GemmArgs& a, int nt, int num_sms, cudaStream_t s);
cudaError_t launch_down(const CUtensorMap& wd, const CUtensorMap& h, const GemmArgs& a, int nt,
                        int num_sms, cudaStream_t s);

}  // namespace beam
