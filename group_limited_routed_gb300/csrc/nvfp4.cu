// NVFP4 experts: E2M1 weights with one E4M3 scale per 16 elements along K and
// one FP32 scale per expert and projection ("SGLang 原生支持 Reflection 的 Beam
// 并驱动其生产 API", section "Highlights": ModelOpt NVFP4 checkpoints; "vLLM 实现
// Reflection Beam 501B MoE 模型 Day 0 支持", section "The fused graph": the NVFP4
// MoE path quantises the activations and runs two grouped GEMMs).
//
// Both GEMM inputs are NVFP4 so the tensor cores run block-scaled FP4 MMAs
// (kind::mxf4nvf4, UE4M3 scales per 16): the token rows x are quantised per
// 16 along d (scale = E4M3(amax / 6), codes = E2M1(x / scale), both with FP32
// divisions, round to nearest even, saturating), and the FP32 SwiGLU product
// h is quantised the same way along d_ff inside the gate/up epilogue.  The
// per-expert FP32 scales multiply the accumulators in the epilogues.
//
// MXFP8 experts share this kernel (FMT = kFmtMxfp8): E4M3 weights with one
// E8M0 scale per 32 elements along K (the OCP MX format; the pages list MXFP8
// beside FP8: "vLLM 实现 Reflection Beam 501B MoE 模型 Day 0 支持", the SkyRL
// paragraphs), both GEMM inputs quantised to MX blocks of 32 (x from its
// BF16 values, h from the FP32 SwiGLU product in the gate/up epilogue) with
// the OCP conversion: shared exponent X = floor(log2(amax)) - 8, codes
// E4M3(v * 2^-X), nearest even, saturating.  The MMAs are
// kind::mxf8f6f4.block_scale (UE8M0, one scale per 32, K = 32 per MMA).  A
// stage holds 128 K values; each row's four scales of a stage (one per MMA)
// sit in one 32-bit TMEM word, and each MMA picks its byte through the scale
// IDs of its instruction descriptor.  The weight scales use the same
// 128-row x 4-scale blocked order as the NVFP4 ones (one 512-byte block per
// stage); the token scales take one 16-byte slot per 128 elements (4 scales,
// then padding).
//
// Scale factors reach the tensor cores through TMEM (tcgen05.cp).  For
// 128 weight rows the MMA wants row r's four scales of a 64-wide K chunk at
// lane r % 32, column base + r / 32: the weight scales are stored in that
// 128-row x 4-scale blocked order (512 bytes per block, made once by
// beam_moe_nvfp4_pack_scales).  Token blocks here have at most 32 rows; the
// token scales are stored per row as one 16-byte slot per 64-wide K chunk
// (its four scales, then padding), so a 32-row x 16-byte copy per chunk puts
// each chunk's scales at its own 4-column-aligned TMEM address.
#include <cuda.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "launch_once.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace beam {
namespace {

using gemm::TileInfo;
using gemm::Waiter;
using gemm::decode_tile;
using gemm::token_blocks;

constexpr unsigned kFull = 0xffffffffu;
constexpr int BM = 128;
constexpr int BK_BYTES = 128;         // K per stage: 256 FP4 or 128 E4M3 elements
constexpr int kMmaBytes = 32;         // K bytes per MMA: 64 FP4 or 32 E4M3 elements
constexpr int kFmtNvfp4 = 0;
constexpr int kFmtMxfp8 = 1;
constexpr int kThreads = 192;
constexpr int kMaxE = 256;
constexpr uint32_t kTileBudget = 216 * 1024;

constexpr uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }
constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// ------------------------------------------------------------ E4M3 / E2M1
__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float e4m3_value(uint8_t c) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(h));
}

__device__ __forceinline__ uint8_t to_e2m1(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp4(v, __NV_E2M1, cudaRoundNearest)) & 0xF;
}

// The shared exponent of an MX block of E4M3 elements: floor(log2(amax)) - 8
// (8 = E4M3's largest exponent), clamped to E8M0's [-127, 127]; -127 when
// amax is 0 or subnormal (floor(log2) < -126 there).  amax >= 0.
__device__ __forceinline__ int mx_exponent(float amax) {
  const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  if (ex == 0) return -127;
  return max(-127, min(127, ex - 127 - 8));
}

// 2^-x as an FP32 for x in [-127, 119] (the exponents mx_exponent returns
// for finite amax): a normal number, so v * 2^-x is exact.
__device__ __forceinline__ float pow2_neg(int x) {
  return __uint_as_float(static_cast<uint32_t>(127 - x) << 23);
}

// ---------------------------------------------------------- pack scales
// [rows, S] row-major E4M3 scales -> 128 x 4 blocks of 512 bytes, block
// (row / 128, s / 4) at ((row / 128) * (S / 4) + s / 4) * 512, inside it
// byte (r % 32) * 16 + (r / 32) * 4 + s % 4 with r = row % 128.
__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t* __restrict__ src,
                                                          int64_t rows, int64_t S,
                                                          uint8_t* __restrict__ dst) {
  const int64_t groups = rows * (S / 4);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < groups;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / (S / 4), sg = i % (S / 4);
    const uint32_t v = *reinterpret_cast<const uint32_t*>(src + row * S + sg * 4);
    const int64_t blk = (row / 128) * (S / 4) + sg;
    const int r = static_cast<int>(row % 128);
    *reinterpret_cast<uint32_t*>(dst + blk * 512 + (r % 32) * 16 + (r / 32) * 4) = v;
  }
}

// ------------------------------------------------------ quantise token rows
// Token t's hidden row, quantised per 16 along d once and written to each of
// its k permuted rows (pair_row[t * k + j]; -1 for an invalid routed index,
// skipped).  xq [rows, d/2] packed E2M1 (low
// nibble = even element); xsf [rows, d/4]: per 64 elements a 16-byte slot
// holding their 4 scales (then padding).
__global__ void __launch_bounds__(128) quantize_tokens_kernel(const uint16_t* __restrict__ x,
                                                              const int32_t* __restrict__ pair_row,
                                                              int32_t k, int32_t d,
                                                              uint8_t* __restrict__ xq,
                                                              uint8_t* __restrict__ xsf,
                                                              uint32_t* status) {
  // programmatic dependent launch: pair_row comes from the permutation just
  // before; once it is visible the gate/up GEMM may start its weight loads
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int64_t t = blockIdx.x;
  __shared__ int64_t s_row[32];
  if (threadIdx.x < k) {
    const int64_t row = pair_row[t * k + threadIdx.x];
    s_row[threadIdx.x] =
        in_bounds(row < static_cast<int64_t>(gridDim.x) * k, status) ? row : -1;
  }
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
  for (int blk = threadIdx.x; blk < d / 16; blk += blockDim.x) {
    const uint4 a = src[2 * blk], b = src[2 * blk + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
    }
    const uint8_t sfc = to_e4m3(__fdiv_rn(amax, 6.0f));
    const float scale = e4m3_value(sfc);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t c = scale > 0.f ? to_e2m1(__fdiv_rn(v[i], scale)) : 0u;
      if (i < 8)
        lo |= c << (4 * i);
      else
        hi |= c << (4 * (i - 8));
    }
    for (int j = 0; j < k; ++j) {
      const int64_t row = s_row[j];
      if (row < 0) continue;  // an invalid routed index has no permuted row
      *reinterpret_cast<uint2*>(xq + row * (d / 2) + blk * 8) = make_uint2(lo, hi);
      xsf[row * (d / 4) + (blk / 4) * 16 + (blk % 4)] = sfc;
    }
  }
}

// Token t's hidden row as MX blocks of 32 along d (E4M3 codes, E8M0 scale),
// quantised once and written to each of its k permuted rows (pair_row[t * k
// + j]; -1 for an invalid routed index, skipped).  xq [rows, d] codes; xsf
// [rows, d/8]: per 128 elements a 16-byte slot holding their 4 scales (then
// padding).  One thread per block of 32.
__global__ void __launch_bounds__(128) quantize_tokens_mx_kernel(const uint16_t* __restrict__ x,
                                                                 const int32_t* __restrict__ pair_row,
                                                                 int32_t k, int32_t d,
                                                                 uint8_t* __restrict__ xq,
                                                                 uint8_t* __restrict__ xsf,
                                                                 uint32_t* status) {
  // as quantize_tokens_kernel
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int64_t t = blockIdx.x;
  __shared__ int64_t s_row[32];
  if (threadIdx.x < k) {
    const int64_t row = pair_row[t * k + threadIdx.x];
    s_row[threadIdx.x] =
        in_bounds(row < static_cast<int64_t>(gridDim.x) * k, status) ? row : -1;
  }
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
  for (int blk = threadIdx.x; blk < d / 32; blk += blockDim.x) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a = src[4 * blk + i];
      w[4 * i] = a.x;
      w[4 * i + 1] = a.y;
      w[4 * i + 2] = a.z;
      w[4 * i + 3] = a.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                               fabsf(__uint_as_float(w[i] & 0xffff0000u))));
    const int xe = mx_exponent(amax);
    const float inv = pow2_neg(xe);
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo0 = to_e4m3(__uint_as_float(w[2 * i] << 16) * inv);
      const uint32_t hi0 = to_e4m3(__uint_as_float(w[2 * i] & 0xffff0000u) * inv);
      const uint32_t lo1 = to_e4m3(__uint_as_float(w[2 * i + 1] << 16) * inv);
      const uint32_t hi1 = to_e4m3(__uint_as_float(w[2 * i + 1] & 0xffff0000u) * inv);
      q[i] = lo0 | (hi0 << 8) | (lo1 << 16) | (hi1 << 24);
    }
    const uint8_t sc = static_cast<uint8_t>(xe + 127);
    for (int j = 0; j < k; ++j) {
      const int64_t row = s_row[j];
      if (row < 0) continue;  // an invalid routed index has no permuted row
      uint4* dst = reinterpret_cast<uint4*>(xq + row * d + 32 * blk);
      dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
      dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
      xsf[row * (d / 8) + (blk / 4) * 16 + (blk % 4)] = sc;
    }
  }
}

// ------------------------------------------------- block-scaled GEMM
// Kinds: the gate/up GEMM (gate and up weight tiles of the same rows, one
// token tile), the down GEMM (one weight tile), and the down GEMM over pairs
// of adjacent 128-row weight blocks sharing one token tile (twice the weight
// bytes per stage for the same per-stage copies and barriers).
constexpr int kKindDown = 0;
constexpr int kKindGateUp = 1;
constexpr int kKindDownPair = 2;

template <int NT, int KIND, int FMT>
struct Cfg {
  static constexpr bool GATEUP = KIND == kKindGateUp;
  static constexpr int NUM_A = KIND == kKindDown ? 1 : 2;
  // 512-byte scale blocks per operand and stage: NVFP4 one per MMA (four
  // scales of 16 per row), MXFP8 one per stage (one scale of 32 per row and
  // MMA, the four MMAs' in one word)
  static constexpr int SBS = FMT == kFmtNvfp4 ? 4 : 1;
  static constexpr uint32_t A_BYTES = BM * BK_BYTES;           // 16 KB
  static constexpr uint32_t B_BYTES = NT * BK_BYTES;
  static constexpr uint32_t SFA_BYTES = 512 * SBS;             // 128 rows x 4 B per block
  static constexpr uint32_t SFB_BYTES = 512 * SBS;             // 32 rows x 16 B per block
  static constexpr uint32_t OFF_B = NUM_A * A_BYTES;
  static constexpr uint32_t OFF_SFA = OFF_B + B_BYTES;
  static constexpr uint32_t OFF_SFB = OFF_SFA + NUM_A * SFA_BYTES;
  static constexpr uint32_t STAGE_BYTES = round_up(OFF_SFB + SFB_BYTES, 1024);
  static constexpr uint32_t TX_BYTES = NUM_A * (A_BYTES + SFA_BYTES) + B_BYTES + SFB_BYTES;
  static constexpr int STAGES_RAW = static_cast<int>(kTileBudget / STAGE_BYTES);
  static constexpr int STAGES = STAGES_RAW > 16 ? 16 : STAGES_RAW;
  static constexpr uint32_t ACC_COLS = NUM_A * NT;
  static constexpr uint32_t SF_COLS = 4 * SBS * (NUM_A + 1);   // one stage's scales
  static constexpr uint32_t SF_BASE = 2 * ACC_COLS;
  static constexpr uint32_t TMEM_COLS = pow2_at_least(SF_BASE + 2 * SF_COLS);
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 5;
  static constexpr uint32_t MISC_BYTES = 16 + 4 * (3 * kMaxE + 1);
  static constexpr uint32_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + MISC_BYTES;
  static_assert(NT == 16 || NT == 32, "token scales are read row-major: at most 32 rows");
  static_assert(B_BYTES % 1024 == 0, "stage alignment");
  static_assert(TMEM_COLS <= 512, "TMEM columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

template <int NT, int KIND, int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    fp4_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0,
                    const __grid_constant__ CUtensorMap tm_a1,
                    const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sfb, const Fp4GemmArgs p) {
  using C = Cfg<NT, KIND, FMT>;
  constexpr bool MX = FMT == kFmtMxfp8;
  constexpr bool GATEUP = C::GATEUP;
  constexpr bool PAIR = KIND == kKindDownPair;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t tiles = raw_addr + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  int32_t* misc = reinterpret_cast<int32_t*>(bars + C::NUM_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int32_t* abort_flag = misc + 1;
  int32_t* s_total = misc + 2;  // permuted rows of all experts (offsets[E])
  int32_t* s_cnt = misc + 4;
  int32_t* s_off = s_cnt + kMaxE;
  int32_t* s_start = s_off + kMaxE;

  const uint32_t bar0 = ptx::smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
  const uint32_t done_bar = bar0 + 8u * (2 * C::STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 128);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    *s_total = p.offsets[E];
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_a0);
    if (GATEUP) ptx::prefetch_tmap(&tm_a1);
    ptx::prefetch_tmap(&tm_b);
    ptx::prefetch_tmap(&tm_sfb);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  for (int e = threadIdx.x; e < E; e += kThreads) {
    s_cnt[e] = p.counts[e];
    s_off[e] = p.offsets[e];
  }
  __syncthreads();
  if (warp == 0) {
    int running = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int v = e < E ? p.m_blocks * token_blocks<NT>(s_cnt[e]) : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) s_start[e] = running + incl - v;
      running += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) s_start[E] = running;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = s_start[E];
  const Waiter W{abort_flag, p.status, p.wait_limit_ns};
  // a tile to work on (see expert_gemm_kernel): rows to process, and (debug
  // build) every index of it inside its buffers, decided alike by every role
  auto use_tile = [&](const TileInfo& ti) {
    if (ti.nvalid <= 0) return false;
    return in_bounds(ti.expert >= 0 && ti.expert < E && ti.mblock >= 0 &&
                         ti.mblock < p.m_blocks && ti.row0 >= 0 &&
                         ti.row0 + ti.nvalid <= *s_total && ti.n_mma <= NT,
                     p.status);
  };
  // weight scales: blocks of 128 rows x 4 scales; a stage takes SBS blocks
  const int64_t sf_blocks_per_row_tile = static_cast<int64_t>(p.k_blocks) * C::SBS;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w =
          p.weight_evict_first ? ptx::policy_evict_first() : ptx::policy_evict_normal();
      const uint64_t pol_b = ptx::policy_evict_last();
      int last_parity[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) last_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // Programmatic dependent launch: the token rows (x or h) come from the
      // kernel before this one, the weights and the tile list do not (the
      // list is the permutation's, complete before that kernel let this one
      // start).  The first tile's first stages get their weight loads before
      // the dependency wait and their token loads after it.
      bool waited = false;
      auto token_loads = [&](int stg, int kb, int b_row0) {
        const uint32_t st = tiles + stg * C::STAGE_BYTES;
        const uint32_t fb = full_bar(stg);
        ptx::tma_load_2d(st + C::OFF_B, &tm_b, fb, kb * BK_BYTES, b_row0, pol_b);
#pragma unroll
        for (int c = 0; c < C::SBS; ++c)
          ptx::tma_load_2d(st + C::OFF_SFB + 512 * c, &tm_sfb, fb, (C::SBS * kb + c) * 16, b_row0,
                           pol_b);
      };
      auto dependency_wait = [&](int npre, int b_row0) {
        ptx::grid_dep_wait();
        ptx::grid_dep_launch();
        waited = true;
        for (int j = 0; j < npre; ++j) token_loads(j, j, b_row0);  // stage j holds K block j
      };
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
        if (!use_tile(ti)) continue;
        int a_row = ti.expert * p.rows_per_expert + ti.mblock * (PAIR ? 2 * BM : BM);
        // the boxes' rows (and so their scale blocks) inside the weight
        // tensor, the token box's first row inside the token operand
        if (!in_bounds(a_row + (PAIR ? 2 * BM : BM) <= p.a_rows, p.status)) a_row = 0;
        const int b_row0 = in_bounds(ti.row0 < p.b_rows, p.status) ? ti.row0 : 0;
        const int64_t sf_row_tile = a_row / BM;
        // the first tile starts at stage 0: its first npre K blocks fill
        // stages 0 .. npre - 1 before the wait
        const int npre = waited ? 0 : min(C::STAGES, p.k_blocks);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!waited && kb == npre) dependency_wait(npre, b_row0);
          if (!W.wait(empty_bar(stage), phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t st = tiles + stage * C::STAGE_BYTES;
          const uint32_t fb = full_bar(stage);
          ptx::mbar_arrive_expect_tx(fb, C::TX_BYTES);
          ptx::tma_load_2d(st, &tm_a0, fb, kb * BK_BYTES, a_row, pol_w);
          const int64_t sf_off = (sf_row_tile * sf_blocks_per_row_tile + C::SBS * kb) * 512;
          ptx::bulk_load(st + C::OFF_SFA, p.sfa0 + sf_off, C::SFA_BYTES, fb);
          if (GATEUP) {
            ptx::tma_load_2d(st + C::A_BYTES, &tm_a1, fb, kb * BK_BYTES, a_row, pol_w);
            ptx::bulk_load(st + C::OFF_SFA + C::SFA_BYTES, p.sfa1 + sf_off, C::SFA_BYTES, fb);
          }
          if (PAIR) {  // the next 128 rows of the same projection
            ptx::tma_load_2d(st + C::A_BYTES, &tm_a0, fb, kb * BK_BYTES, a_row + BM, pol_w);
            ptx::bulk_load(st + C::OFF_SFA + C::SFA_BYTES,
                           p.sfa0 + sf_off + sf_blocks_per_row_tile * 512, C::SFA_BYTES, fb);
          }
          if (waited) token_loads(stage, kb, b_row0);
          last_parity[stage] = static_cast<int>(phase);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        // a first tile of at most STAGES K blocks: its token loads follow here
        if (ok && !waited) dependency_wait(npre, b_row0);
      }
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s)
        if (last_parity[s] >= 0) W.wait_final(full_bar(s), static_cast<uint32_t>(last_parity[s]));
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int sf_slot = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
        if (!use_tile(ti)) continue;
        const uint32_t idesc = MX ? ptx::idesc_mx8_f32(BM, static_cast<uint32_t>(ti.n_mma))
                                  : ptx::idesc_fp4_f32(BM, static_cast<uint32_t>(ti.n_mma));
        if (!W.wait(tempty_bar(acc), acc_phase ^ 1u)) break;
        ptx::tc_fence_after();
        // the accumulators below the scale columns
        in_bounds(acc * C::ACC_COLS + C::NUM_A * ti.n_mma <= C::SF_BASE, p.status);
        const uint32_t d0 = tmem_base + acc * C::ACC_COLS;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!W.wait(full_bar(stage), phase)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st = tiles + stage * C::STAGE_BYTES;
          const uint32_t sf_col = tmem_base + C::SF_BASE + sf_slot * C::SF_COLS;
          // scales of this stage into TMEM (in issue order with the MMAs):
          // each 512-byte block to 4 columns
#pragma unroll
          for (int a = 0; a < C::NUM_A; ++a)
#pragma unroll
            for (int c = 0; c < C::SBS; ++c)
              ptx::tmem_cp_32x128b_x4(sf_col + 4 * C::SBS * a + 4 * c,
                                      ptx::sdesc_rows16(st + C::OFF_SFA + a * C::SFA_BYTES + 512 * c));
          const uint32_t sfb_col = sf_col + 4 * C::SBS * C::NUM_A;
#pragma unroll
          for (int c = 0; c < C::SBS; ++c)
            ptx::tmem_cp_32x128b_x4(sfb_col + 4 * c, ptx::sdesc_rows16(st + C::OFF_SFB + 512 * c));
#pragma unroll
          for (int c = 0; c < BK_BYTES / kMmaBytes; ++c) {
            const uint32_t accum = (kb | c) ? 1u : 0u;
            const uint64_t bd = ptx::sdesc_sw128(st + C::OFF_B + kMmaBytes * c);
            if constexpr (MX) {
              // MMA c takes byte c of each row's scale word
              const uint32_t id = idesc | ptx::idesc_sf_ids(c, c);
              ptx::mma_mx8(d0, ptx::sdesc_sw128(st + kMmaBytes * c), bd, id, sf_col, sfb_col, accum);
              if (C::NUM_A == 2)
                ptx::mma_mx8(d0 + NT, ptx::sdesc_sw128(st + C::A_BYTES + kMmaBytes * c), bd, id,
                             sf_col + 4, sfb_col, accum);
            } else {
              ptx::mma_fp4(d0, ptx::sdesc_sw128(st + kMmaBytes * c), bd, idesc, sf_col + 4 * c,
                           sfb_col + 4 * c, accum);
              if (C::NUM_A == 2)
                ptx::mma_fp4(d0 + NT, ptx::sdesc_sw128(st + C::A_BYTES + kMmaBytes * c), bd, idesc,
                             sf_col + 16 + 4 * c, sfb_col + 4 * c, accum);
            }
          }
          ptx::mma_commit(empty_bar(stage));
          sf_slot ^= 1;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(tfull_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      ptx::mma_commit(done_bar);
      W.wait_final(done_bar, 0);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int m = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
      if (!use_tile(ti)) continue;
      if (!W.wait(tfull_bar(acc), acc_phase)) break;
      ptx::tc_fence_after();
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS;
      const int col = ti.mblock * BM + m;
      const float gs0 = MX ? 1.f : p.gs0[ti.expert];
#pragma unroll 1
      for (int c0 = 0; c0 < ti.nvalid; c0 += 16) {
        // the chunk's TMEM columns inside its accumulator
        if (!in_bounds(c0 + 16 <= NT, p.status)) break;
        uint32_t ra[16];
        ptx::tmem_ld16(tq + c0, ra);
        if constexpr (GATEUP && MX) {
          uint32_t rb[16];
          ptx::tmem_ld16(tq + NT + c0, rb);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {  // uniform across the warp
              const int64_t row = ti.row0 + c0 + j;
              // uniform too (the shuffles below need every lane)
              if (!in_bounds(row < p.out_rows_cap && (ti.mblock + 1) * BM <= p.out_ld, p.status))
                continue;
              const float g = __uint_as_float(ra[j]);
              const float u = __uint_as_float(rb[j]);
              const float h = g / (1.0f + expf(-g)) * u;
              // an MX block of 32 along d_ff: the warp's 32 lanes
              float amax = fabsf(h);
#pragma unroll
              for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
              const int xe = mx_exponent(amax);
              p.hq[row * p.out_ld + col] = to_e4m3(h * pow2_neg(xe));
              if (lane == 0)
                p.hsf[row * (p.out_ld / 8) + (col / 128) * 16 + (col / 32) % 4] =
                    static_cast<uint8_t>(xe + 127);
            }
          }
        } else if constexpr (GATEUP) {
          const float gs1 = p.gs1[ti.expert];
          uint32_t rb[16];
          ptx::tmem_ld16(tq + NT + c0, rb);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {  // uniform across the warp
              const int64_t row = ti.row0 + c0 + j;
              if (!in_bounds(row < p.out_rows_cap && (ti.mblock + 1) * BM <= p.out_ld, p.status))
                continue;
              const float g = __uint_as_float(ra[j]) * gs0;
              const float u = __uint_as_float(rb[j]) * gs1;
              const float h = g / (1.0f + expf(-g)) * u;
              // NVFP4 along d_ff: 16 consecutive f = 16 lanes
              float amax = fabsf(h);
#pragma unroll
              for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
              const uint8_t sfc = to_e4m3(__fdiv_rn(amax, 6.0f));
              const float scale = e4m3_value(sfc);
              const uint32_t code = scale > 0.f ? to_e2m1(__fdiv_rn(h, scale)) : 0u;
              const uint32_t other = __shfl_xor_sync(kFull, code, 1);
              if ((lane & 1) == 0)
                p.hq[row * (p.out_ld / 2) + col / 2] = static_cast<uint8_t>(code | (other << 4));
              if ((lane & 15) == 0)
                p.hsf[row * (p.out_ld / 4) + (col / 64) * 16 + (col / 16) % 4] = sfc;
            }
          }
        } else if constexpr (PAIR) {
          uint32_t rb[16];
          ptx::tmem_ld16(tq + NT + c0, rb);
          ptx::tmem_wait_ld();
          // this pair's first 128 rows are output columns col, the next col + 128
          const int pcol = ti.mblock * 2 * BM + m;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {
              const int row = ti.row0 + c0 + j;
              const int orow = p.out_rows ? p.out_rows[row] : row;
              if (!in_bounds(orow >= 0 && orow < p.out_rows_cap && pcol + BM < p.out_ld,
                             p.status))
                continue;
              const float wr = gs0 * p.perm_w[row];
              p.y[static_cast<int64_t>(orow) * p.out_ld + pcol] = __uint_as_float(ra[j]) * wr;
              p.y[static_cast<int64_t>(orow) * p.out_ld + pcol + BM] = __uint_as_float(rb[j]) * wr;
            }
          }
        } else {
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {
              const int row = ti.row0 + c0 + j;
              if (!in_bounds(row < p.out_rows_cap && col < p.out_ld, p.status)) continue;
              p.y[static_cast<int64_t>(row) * p.out_ld + col] =
                  __uint_as_float(ra[j]) * gs0 * p.perm_w[row];
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int NT, int KIND, int FMT>
cudaError_t launch_fp4_impl(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                            const CUtensorMap& sfb, const Fp4GemmArgs& p, int grid,
                            cudaStream_t s) {
  using C = Cfg<NT, KIND, FMT>;
  const cudaError_t err = smem_limit_once<fp4_gemm_kernel<NT, KIND, FMT>>(C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  return launch_dependent(fp4_gemm_kernel<NT, KIND, FMT>, dim3(grid), dim3(kThreads), C::SMEM_BYTES,
                          s, a0, a1, b, sfb, p);
}

}  // namespace

void launch_pack_scales(const uint8_t* src, int64_t rows, int64_t S, uint8_t* dst,
                        cudaStream_t s) {
  const int64_t groups = rows * (S / 4);
  const int grid = static_cast<int>((groups + 255) / 256 < 4096 ? (groups + 255) / 256 : 4096);
  pack_scales_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(src, rows, S, dst);
}

void launch_quantize_tokens(const uint16_t* x, const int32_t* pair_row, int64_t T, int32_t k,
                            int32_t d, uint8_t* xq, uint8_t* xsf, uint32_t* status,
                            cudaStream_t s) {
  if (T <= 0) return;
  launch_dependent(quantize_tokens_kernel, dim3(static_cast<unsigned>(T)), dim3(128), 0, s, x,
                   pair_row, k, d, xq, xsf, status);
}

cudaError_t launch_fp4_gemm(bool gateup, int nt, const CUtensorMap& a0, const CUtensorMap& a1,
                            const CUtensorMap& b, const CUtensorMap& sfb, const Fp4GemmArgs& p,
                            int grid, cudaStream_t s) {
  // the down GEMM takes weight rows in pairs of 128-row blocks (m_blocks
  // counts pairs)
  if (gateup) {
    if (nt == 16) return launch_fp4_impl<16, kKindGateUp, kFmtNvfp4>(a0, a1, b, sfb, p, grid, s);
    if (nt == 32) return launch_fp4_impl<32, kKindGateUp, kFmtNvfp4>(a0, a1, b, sfb, p, grid, s);
  } else {
    if (nt == 16) return launch_fp4_impl<16, kKindDownPair, kFmtNvfp4>(a0, a0, b, sfb, p, grid, s);
    if (nt == 32) return launch_fp4_impl<32, kKindDownPair, kFmtNvfp4>(a0, a0, b, sfb, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

void launch_quantize_tokens_mx(const uint16_t* x, const int32_t* pair_row, int64_t T, int32_t k,
                               int32_t d, uint8_t* xq, uint8_t* xsf, uint32_t* status,
                               cudaStream_t s) {
  if (T <= 0) return;
  launch_dependent(quantize_tokens_mx_kernel, dim3(static_cast<unsigned>(T)), dim3(128), 0, s, x,
                   pair_row, k, d, xq, xsf, status);
}

cudaError_t launch_mxfp8_gemm(bool gateup, int nt, const CUtensorMap& a0, const CUtensorMap& a1,
                              const CUtensorMap& b, const CUtensorMap& sfb, const Fp4GemmArgs& p,
                              int grid, cudaStream_t s) {
  if (gateup) {
    if (nt == 16) return launch_fp4_impl<16, kKindGateUp, kFmtMxfp8>(a0, a1, b, sfb, p, grid, s);
    if (nt == 32) return launch_fp4_impl<32, kKindGateUp, kFmtMxfp8>(a0, a1, b, sfb, p, grid, s);
  } else {
    if (nt == 16) return launch_fp4_impl<16, kKindDownPair, kFmtMxfp8>(a0, a0, b, sfb, p, grid, s);
    if (nt == 32) return launch_fp4_impl<32, kKindDownPair, kFmtMxfp8>(a0, a0, b, sfb, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace beam
