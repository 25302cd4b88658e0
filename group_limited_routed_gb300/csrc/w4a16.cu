// NVFP4 experts with 16-bit activations (W4A16): the weights stay E2M1 with
// one E4M3 scale per 16 along K and one FP32 scale per expert and projection
// ("SGLang 原生支持 Reflection 的 Beam 并驱动其生产 API", section "Highlights":
// ModelOpt NVFP4 checkpoints), the activations are not quantised.
//
// The tensor cores take F16 operands here (kind::f16 with F16 A and B):
//   - a weight E2M1 code times its E4M3 scale has at most 6 significant bits
//     and lies in [2^-10, 2688], so it is exact in F16; the FP32 expert scale
//     multiplies the accumulator in the epilogue;
//   - the token rows x (BF16) are converted to F16 when they are gathered
//     (exact inside F16's normal range, saturating at 65504), and the SwiGLU
//     product h is rounded to F16 for the down GEMM.
// The weight tiles stay packed in shared memory (0.5 byte per weight); eight
// converter warps (two per TMEM lane quarter, taking alternate 64-wide K
// slices whole) expand each row's K slice of both weight tiles of a stage
// to F16 pairs in registers and store it into tensor memory, where the MMA
// reads its A operand.  So shared memory carries only the packed codes and
// the token tiles.  A stage holds two weight tiles: gate and up, or for the
// down GEMM two adjacent 128-row blocks of W_d that share the token tile.
//
// At decode-sized batches this path issues many tiny MMAs: an F16 MMA covers
// K = 16 per instruction (the block-scaled FP4 MMA of the NVFP4 path covers
// 64), and a few token rows per expert keep N at 16.  Four threads issue
// them, each into its own accumulator (see kIssuers).
#include <cuda.h>
#include <cuda_fp16.h>
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
constexpr int KS_BYTES = 128;  // 256 E2M1 codes of K per row and stage
constexpr int KSUB = 64;       // K per converted slice: 32 TMEM columns of F16 pairs
constexpr int kMaxE = 256;
constexpr int kConvWarps = 8;  // two per TMEM lane quarter, each half of a K slice
constexpr int kEpiWarp0 = 2 + kConvWarps;             // first of the 4 epilogue warps
// warps: producer, MMA issuer, converters, epilogue, and three more MMA
// issuers (warps 14-16).  kIssuers threads issue the MMAs, each into its own
// accumulator: for gate/up, issuer i takes projection i % 2 and one of
// kIssuers / 2 parts of every K slice; for down, one of kIssuers parts.  The
// epilogue adds the partial sums in issuer order.  At a few token rows per
// expert the tiny MMAs are issue-bound: one thread alone leaves the tensor
// pipe idle (four issuers: gate/up 1051 -> 748 us, down 760 -> 559 us on
// the 128-token NVFP4 batch; eight gave no more).
constexpr int kIssuers = 4;
// Kernel modes: gate/up (W_g and W_u tiles of the same rows), down over two
// adjacent 128-row W_d blocks that share the token tile (the two blocks take
// the places of gate and up; m_blocks = d / 256, d % 256 == 0 for NVFP4).
// The two converter warps of a lane quarter take alternate 64-wide slices
// whole: a warp's TMEM stores wait behind the queued MMAs, and the other warp
// converts meanwhile (gate/up 747 -> 709 us on the 128-token batch; the down
// GEMM over single 128-row blocks, with half of every slice per warp, took
// 569 us against 377 us over pairs of blocks).
constexpr int kW4GateUp = 1;
constexpr int kW4DownPair = 2;
constexpr int kIssuer1 = kEpiWarp0 + 4;  // warps of issuers 1..kIssuers-1
constexpr int kThreads = 32 * (kIssuer1 + kIssuers - 1);
constexpr uint32_t kTileBudget = 216 * 1024;

constexpr uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }
constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int NT, int MODE>
struct Cfg {
  static constexpr int NUM_A = 2;
  static constexpr int NUM_ACC = kIssuers;  // one accumulator per issuer
  static constexpr uint32_t A_BYTES = BM * KS_BYTES;     // 16 KB of codes per projection
  static constexpr uint32_t SFA_BYTES = 2048;            // 4 blocks of 128 rows x 4 scales
  static constexpr uint32_t B_SUB = NT * KSUB * 2;       // one 64-wide K slice of F16 rows
  static constexpr uint32_t OFF_SFA = NUM_A * A_BYTES;
  static constexpr uint32_t OFF_B = OFF_SFA + NUM_A * SFA_BYTES;
  static constexpr uint32_t STAGE_BYTES = round_up(OFF_B + 4 * B_SUB, 1024);
  static constexpr uint32_t TX_BYTES = NUM_A * (A_BYTES + SFA_BYTES) + 4 * B_SUB;
  static constexpr int STAGES_RAW = static_cast<int>(kTileBudget / STAGE_BYTES);
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr uint32_t ACC_COLS = NUM_ACC * NT;
  static constexpr uint32_t A_COLS = NUM_A * (KSUB / 2);  // one converted slice
  static constexpr uint32_t A_BASE = 2 * ACC_COLS;
  // converted slices in flight: four.  Each converter warp's TMEM stores
  // wait behind the MMAs already queued, so a deeper ring lengthens that
  // wait (128-token NVFP4 batch: 6 slots 1.190 ms per layer, 4 slots
  // 1.142 ms, 2 slots 1.167 ms)
  static constexpr int RA_RAW = static_cast<int>((512 - A_BASE) / A_COLS);
  static constexpr int RA = 4;
  static constexpr uint32_t TMEM_COLS = pow2_at_least(A_BASE + RA * A_COLS);
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 * RA + 5;
  static constexpr uint32_t MISC_BYTES = 16 + 4 * (3 * kMaxE + 1);
  static constexpr uint32_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + MISC_BYTES;
  static_assert(OFF_B % 1024 == 0 && B_SUB % 1024 == 0, "token tiles keep 1024-byte alignment");
  static_assert(NT == 16 || NT == 32, "token block width");
  static_assert(TMEM_COLS <= 512, "TMEM columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(STAGES >= 2, "two stages at least");
  static_assert(RA <= RA_RAW, "TMEM holds the accumulators and RA converted slices");
  static_assert(RA % 2 == 0,
                "slices alternate between two converter warps: an even ring");
};

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// kind::f16 MMA whose A operand (M = 128 rows, one per lane; column j holds
// K elements 2j and 2j+1 in its low and high halves) is in tensor memory.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::f16 with F16 A and B (format 0), FP32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ uint16_t f32_to_f16_sat(float v) {
  v = fminf(fmaxf(v, -65504.0f), 65504.0f);
  return __half_as_ushort(__float2half_rn(v));
}

// 4 packed bytes (8 codes, low nibble = even element) -> 4 F16 pairs, each
// times the F16 pair s2: the word is split into its bytes in one move and
// each byte goes through the hardware E2M1x2 -> F16x2 conversion.
__device__ __forceinline__ void dequant8(uint32_t codes, uint32_t s2, uint32_t* out) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 h0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
      "mul.rn.f16x2 %0, h0, %5;\n\t"
      "mul.rn.f16x2 %1, h1, %5;\n\t"
      "mul.rn.f16x2 %2, h2, %5;\n\t"
      "mul.rn.f16x2 %3, h3, %5;\n\t}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(codes), "r"(s2));
}

// an E4M3 scale as an F16 pair (exact: E4M3 values are F16 values)
__device__ __forceinline__ uint32_t scale_pair(uint8_t sf) {
  const __half_raw s = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(sf), __NV_E4M3);
  return static_cast<uint32_t>(s.x) | (static_cast<uint32_t>(s.x) << 16);
}

// ------------------------------------------------------- gather to F16
// x16[row] = f16(x[token of row]) for the permuted rows.
__global__ void __launch_bounds__(128) gather_f16_kernel(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ perm_src,
                                                         const int32_t* __restrict__ n_valid,
                                                         int32_t k, int32_t d,
                                                         uint16_t* __restrict__ x16) {
  // programmatic dependent launch: perm_src and n_valid come from the
  // permutation just before; once they are visible the gate/up GEMM may
  // start its weight loads
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int64_t row = blockIdx.x;
  if (row >= *n_valid) return;
  const int64_t t = perm_src[row] / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
  uint4* dst = reinterpret_cast<uint4*>(x16 + row * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
    const uint4 a = src[i];
    const uint32_t in[4] = {a.x, a.y, a.z, a.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(in[j] << 16), hi = __uint_as_float(in[j] & 0xffff0000u);
      o[j] = static_cast<uint32_t>(f32_to_f16_sat(lo)) |
             (static_cast<uint32_t>(f32_to_f16_sat(hi)) << 16);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------- GEMM
template <int NT, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0,
                      const __grid_constant__ CUtensorMap tm_a1,
                      const __grid_constant__ CUtensorMap tm_b, const W4a16GemmArgs p) {
  using C = Cfg<NT, MODE>;
  constexpr bool GATEUP = MODE == kW4GateUp;
  constexpr bool PAIR = MODE == kW4DownPair;
  static_assert(GATEUP || PAIR, "kernel mode");
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
  auto afull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + C::RA + a); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 * C::RA + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 * C::RA + 2 + a); };
  const uint32_t done_bar = bar0 + 8u * (2 * C::STAGES + 2 * C::RA + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;
  constexpr int NI = kIssuers;  // MMA-issuing threads, each committing its own MMAs

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), NI + kConvWarps);  // the MMA commits and the converters
    }
    for (int a = 0; a < C::RA; ++a) {
      ptx::mbar_init(afull_bar(a), kConvWarps / 2);
      ptx::mbar_init(aempty_bar(a), NI);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), NI);
      ptx::mbar_init(tempty_bar(a), 128);
    }
    ptx::mbar_init(done_bar, NI);
    *abort_flag = 0;
    *s_total = p.offsets[E];
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_a0);
    if (GATEUP) ptx::prefetch_tmap(&tm_a1);
    ptx::prefetch_tmap(&tm_b);
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
  if (warp == 0) {  // exclusive scan of tiles per expert
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
  const int64_t sf_blocks_per_row_tile = p.k_blocks * 4;
  // a tile to work on (see expert_gemm_kernel): rows to process, and (debug
  // build) every index of it inside its buffers, decided alike by every role
  auto use_tile = [&](const TileInfo& ti) {
    if (ti.nvalid <= 0) return false;
    return in_bounds(ti.expert >= 0 && ti.expert < E && ti.mblock >= 0 &&
                         ti.mblock < p.m_blocks && ti.row0 >= 0 &&
                         ti.row0 + ti.nvalid <= *s_total && ti.n_mma <= NT,
                     p.status);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
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
      // Programmatic dependent launch, as in the NVFP4 GEMM: the token rows
      // come from the kernel before this one; the first tile's first stages
      // get their weight loads before the dependency wait, their token loads
      // after it.
      bool waited = false;
      auto token_loads = [&](int stg, int kb, int b_row0) {
        const uint32_t st = tiles + stg * C::STAGE_BYTES;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ptx::tma_load_2d(st + C::OFF_B + j * C::B_SUB, &tm_b, full_bar(stg), (4 * kb + j) * KSUB,
                           b_row0, pol_b);
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
          ptx::tma_load_2d(st, &tm_a0, fb, kb * KS_BYTES, a_row, pol_w);
          const int64_t sf_off = (sf_row_tile * sf_blocks_per_row_tile + 4 * kb) * 512;
          ptx::bulk_load(st + C::OFF_SFA, p.sfa0 + sf_off, C::SFA_BYTES, fb);
          if (GATEUP) {
            ptx::tma_load_2d(st + C::A_BYTES, &tm_a1, fb, kb * KS_BYTES, a_row, pol_w);
            ptx::bulk_load(st + C::OFF_SFA + C::SFA_BYTES, p.sfa1 + sf_off, C::SFA_BYTES, fb);
          }
          if (PAIR) {  // the next 128-row block and its scales (the next row tile)
            ptx::tma_load_2d(st + C::A_BYTES, &tm_a0, fb, kb * KS_BYTES, a_row + BM, pol_w);
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
  } else if (warp == 1 || warp >= kIssuer1) {
    // --------------------------------------------------------- MMA issuers
    // issuer i (warp 1 for i = 0, then warps 14, 15, 16) accumulates into
    // accumulator i: weight tile i % 2 (gate or up; the first or second W_d
    // block) and K part i / 2 of each slice
    const int issuer = warp == 1 ? 0 : warp - kIssuer1 + 1;
    if (lane == 0) {
      int stage = 0, ra = 0;
      uint32_t phase = 0, ra_phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
        if (!use_tile(ti)) continue;
        const uint32_t idesc = idesc_f16_f32(BM, static_cast<uint32_t>(ti.n_mma));
        if (!W.wait(tempty_bar(acc), acc_phase ^ 1u)) break;
        ptx::tc_fence_after();
        const uint32_t d0 = tmem_base + acc * C::ACC_COLS;
        for (int kb = 0; ok && kb < p.k_blocks; ++kb) {
          if (!W.wait(full_bar(stage), phase)) {
            ok = false;
            break;
          }
          const uint32_t st = tiles + stage * C::STAGE_BYTES;
          for (int j = 0; j < 4; ++j) {
            if (!W.wait(afull_bar(ra), ra_phase)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t a0 = tmem_base + C::A_BASE + ra * C::A_COLS;
            // this issuer's K steps (of the slice's four) and projection
            constexpr int PARTS = kIssuers / 2;
            constexpr int KK = (KSUB / 16) / PARTS;
            const int proj = issuer % 2;
            const int part = issuer / 2;
#pragma unroll
            for (int i = 0; i < KK; ++i) {
              const int kk = part * KK + i;
              const uint32_t accum = (kb | j | i) ? 1u : 0u;
              const uint64_t bd = ptx::sdesc_sw128(st + C::OFF_B + j * C::B_SUB + kk * 32);
              const uint32_t a_col = a0 + proj * (KSUB / 2) + kk * 8;
              mma_f16_tmem_a(d0 + issuer * NT, a_col, bd, idesc, accum);
            }
            ptx::mma_commit(aempty_bar(ra));
            if (++ra == C::RA) {
              ra = 0;
              ra_phase ^= 1u;
            }
          }
          if (!ok) break;
          ptx::mma_commit(empty_bar(stage));
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
  } else if (warp < kEpiWarp0) {
    // ----------------------------------------------------------- converters
    // Thread row m (its warp's TMEM lane quarter) expands its row's 64-wide
    // K slice j of both weight tiles: per tile 32 code bytes (chunks 2j and
    // 2j + 1 of the 128-byte swizzled row) and 4 scales (blocked order) ->
    // 32 F16 pairs -> 32 TMEM columns.
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;  // which of the two converter warps of lane quarter q
    const int m = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    // global index of this warp's next slice: the slices alternate between
    // the two warps of a lane quarter, each converting whole slices
    uint32_t gs = static_cast<uint32_t>(grp);
    constexpr int JSTEP = 2;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
      if (!use_tile(ti)) continue;
      for (int kb = 0; ok && kb < p.k_blocks; ++kb) {
        if (!W.wait(full_bar(stage), phase)) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + stage * C::STAGE_BYTES;
        for (int j = grp; j < 4; j += JSTEP) {
          const int slot = static_cast<int>(gs % C::RA);
          const uint32_t sph = (gs / C::RA) & 1u;
          if (!W.wait(aempty_bar(slot), sph ^ 1u)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int a = 0; a < C::NUM_A; ++a) {
            const uint8_t* row = st + a * C::A_BYTES + m * KS_BYTES;
            // the slice's four scales of row m (blocked order)
            const uint32_t sf4 = *reinterpret_cast<const uint32_t*>(
                st + C::OFF_SFA + a * C::SFA_BYTES + j * 512 + (m & 31) * 16 + (m >> 5) * 4);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint4 c =
                  *reinterpret_cast<const uint4*>(row + (((2 * j + half) ^ (m & 7)) << 4));
              const uint32_t s0 = scale_pair(static_cast<uint8_t>(sf4 >> (16 * half)));
              const uint32_t s1 = scale_pair(static_cast<uint8_t>(sf4 >> (16 * half + 8)));
              uint32_t v[16];
              dequant8(c.x, s0, v);
              dequant8(c.y, s0, v + 4);
              dequant8(c.z, s1, v + 8);
              dequant8(c.w, s1, v + 12);
              tmem_st16(tmem_base + lane_off + C::A_BASE + slot * C::A_COLS + a * (KSUB / 2) +
                            16 * half,
                        v);
            }
          }
          tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(afull_bar(slot));
          gs += JSTEP;
        }
        if (!ok) break;
        // this stage's codes and scales have been read
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty_bar(stage));
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
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
      const int col = ti.mblock * (PAIR ? 2 * BM : BM) + m;
      const float gs0 = p.gs0[ti.expert];
#pragma unroll 1
      for (int c0 = 0; c0 < ti.nvalid; c0 += 16) {
        // the chunk's TMEM columns inside its accumulators
        if (!in_bounds(c0 + 16 <= NT, p.status)) break;
        // the issuers' partial sums, added in issuer order
        uint32_t r[kIssuers][16];
#pragma unroll
        for (int i = 0; i < kIssuers; ++i) ptx::tmem_ld16(tq + i * NT + c0, r[i]);
        ptx::tmem_wait_ld();
        if constexpr (GATEUP) {
          const float gs1 = p.gs1[ti.expert];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {
              if (!in_bounds(ti.row0 + c0 + j < p.out_rows_cap && col < p.out_ld, p.status))
                continue;
              float ga = __uint_as_float(r[0][j]), ua = __uint_as_float(r[1][j]);
#pragma unroll
              for (int i = 2; i < kIssuers; i += 2) {
                ga += __uint_as_float(r[i][j]);
                ua += __uint_as_float(r[i + 1][j]);
              }
              const float g = ga * gs0;
              const float u = ua * gs1;
              const float h = __fdividef(g, 1.0f + __expf(-g)) * u;
              p.h_out[static_cast<int64_t>(ti.row0 + c0 + j) * p.out_ld + col] = f32_to_f16_sat(h);
            }
          }
        } else {
          // block b's partial sums: issuers b, b + 2, ... in issuer order
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {
              const int row = ti.row0 + c0 + j;
              if (!in_bounds(row < p.out_rows_cap && col + BM < p.out_ld, p.status)) continue;
              const float wr = p.perm_w[row];
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                float acc = __uint_as_float(r[b][j]);
#pragma unroll
                for (int i = b + 2; i < kIssuers; i += 2) acc += __uint_as_float(r[i][j]);
                p.y_out[static_cast<int64_t>(row) * p.out_ld + col + b * BM] = acc * gs0 * wr;
              }
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

template <int NT, int MODE>
cudaError_t launch_impl(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                        const W4a16GemmArgs& p, int grid, cudaStream_t s) {
  using C = Cfg<NT, MODE>;
  const cudaError_t err = smem_limit_once<w4a16_gemm_kernel<NT, MODE>>(C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  return launch_dependent(w4a16_gemm_kernel<NT, MODE>, dim3(grid), dim3(kThreads), C::SMEM_BYTES, s,
                          a0, a1, b, p);
}

}  // namespace

void launch_gather_f16(const uint16_t* x, const int32_t* perm_src, const int32_t* n_valid,
                       int64_t TK, int32_t k, int32_t d, uint16_t* x16, cudaStream_t s) {
  launch_dependent(gather_f16_kernel, dim3(static_cast<unsigned>(TK)), dim3(128), 0, s, x, perm_src,
                   n_valid, k, d, x16);
}

cudaError_t launch_w4a16_gemm(bool gateup, int nt, const CUtensorMap& a0, const CUtensorMap& a1,
                              const CUtensorMap& b, const W4a16GemmArgs& p, int grid,
                              cudaStream_t s) {
  if (gateup) {
    if (nt == 16) return launch_impl<16, kW4GateUp>(a0, a1, b, p, grid, s);
    if (nt == 32) return launch_impl<32, kW4GateUp>(a0, a1, b, p, grid, s);
  } else {
    if (nt == 16) return launch_impl<16, kW4DownPair>(a0, a0, b, p, grid, s);
    if (nt == 32) return launch_impl<32, kW4DownPair>(a0, a0, b, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace beam
