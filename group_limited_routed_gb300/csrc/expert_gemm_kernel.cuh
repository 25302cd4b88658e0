// Device code of the grouped expert GEMMs (launched from expert_gemm.cu,
// the one file that includes this header).
//
// Grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM), operands
// staged by TMA.  One kernel template, two epilogues:
//
//   gate/up : for every expert e and every row r of its permuted tokens,
//             g = x_r W_g[e]^T, u = x_r W_u[e]^T (FP32 accumulators in TMEM),
//             h_r = bf16(silu(g) * u) with the SwiGLU product in FP32
//             ("Reflection 发布 501B 开源模型 Beam，Apache 2.0 许可", section
//             "残差流": the SwiGLU product is computed in FP32; SGLang post
//             "SGLang 原生支持 Reflection 的 Beam 并驱动其生产 API", section "BF16 MoE
//             Kernel Optimization": the activation keeps its BF16 rounding).
//   down    : y_r = w_r * (h_r W_d[e]^T) in FP32 (the FP32 routing weight is
//             applied before anything is rounded; the BF16 rounding happens
//             once, after the local sum over a token's experts -- SGLang post,
//             section "Fusion Optimizations").
//
// Tiling ("swap AB"): the MMA's M side is 128 weight rows, its N side a block
// of the expert's permuted token rows (up to NT; the MMA's N is the block's
// row count rounded up to 16), K steps of one 128-byte swizzle row: 64 BF16
// values, or 128 E4M3 values for the FP8 experts (kind::f8f6f4 MMAs; the
// epilogue then multiplies each accumulator by its weight row's and its
// token row's FP32 scales).  gate/up issue two MMAs per K step into two TMEM accumulators (gate,
// up) that share the token operand, so one thread holds g and u of the same
// (f, token) and the SwiGLU epilogue is local.  An expert's rows are split
// into ceil(rows / NT) blocks of nearly equal size.  With 16-row token
// blocks (decode-sized batches) gate/up gathers its token rows from the
// hidden states with per-row TMA loads, so no permuted copy of x is made;
// rows past a block's last valid row are not loaded and the MMA columns they
// feed are never read.  Larger blocks read a gathered copy of x with tile
// loads (hundreds of 128-byte TMA requests per stage would starve the MMA).
//
// Persistent CTAs (one per SM) walk a tile list derived on the device from
// the per-expert row counts: tile -> (expert, weight block, token block),
// ordered so the token blocks of one weight block run on neighbouring CTAs at
// the same time (their weight tiles are then read from HBM once and from L2
// after).  Warp roles: warp 0 streams weight tiles and warp 2 token tiles,
// each into its own ring, warp 1 owns TMEM and issues tcgen05.mma from one
// thread, the remaining warps drain the accumulators: 4, or for 256-row token
// blocks 8 (down) or 16 (gate/up, whose two accumulators fill TMEM, so the
// MMA waits for this epilogue), several per TMEM lane quarter, each draining
// its share of the columns.  Accumulators are double-buffered when two fit
// in TMEM's 512 columns.  Every
// mbarrier wait is bounded: when one runs out the CTA latches
// BEAM_ERR_TIMEOUT, stops, lets its copies in flight land, frees its TMEM and
// returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "expert_gemm.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace beam {
namespace {

using gemm::TileInfo;
using gemm::Waiter;
using gemm::block_rows;
using gemm::decode_tile;
using gemm::token_blocks;

constexpr unsigned kFull = 0xffffffffu;
constexpr int BM = 128;
constexpr int kRowBytes = 128;     // one K block of one operand row: a 128-byte swizzle row
constexpr int kMmaKBytes = 32;     // K bytes per MMA instruction (16 BF16 or 32 E4M3)
// warps: weight producer, MMA issuer, token producer, then the epilogue warps
// (four per TMEM lane quarter for the single-buffered 256-token gate/up tile,
// whose epilogue the MMA waits for)
constexpr int epi_warps_for(int nt, int mode) {
  return nt >= 256 ? (mode == kModeDown ? 8 : 16) : 4;
}
constexpr int threads_for(int nt, int mode) { return 96 + 32 * epi_warps_for(nt, mode); }
constexpr int kMaxE = 256;
constexpr uint32_t kTileBudget = 216 * 1024;

constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// Two rings of equal depth, one per producer warp: weight tiles and token
// tiles (both may come from HBM: the gathered token copy and h are far larger
// than L2), as many stages as fit.
template <int NT, int MODE>
struct Cfg {
  // gate/up: gate and up tiles of the same rows; down pair: two adjacent
  // 128-row blocks of W_d; both share the token tile
  static constexpr int NUM_A = MODE == kModeDown ? 1 : 2;
  static constexpr uint32_t A_BYTES = BM * kRowBytes;
  static constexpr uint32_t A_STAGE = NUM_A * A_BYTES;
  static constexpr uint32_t B_STAGE = NT * kRowBytes;
  static constexpr int SA_RAW = static_cast<int>(kTileBudget / (A_STAGE + B_STAGE));
  static constexpr int SA = SA_RAW > 16 ? 16 : SA_RAW;
  static constexpr int SB = SA;
  static constexpr uint32_t B_RING = SA * A_STAGE;               // offset of the token ring
  static constexpr int EPI_WARPS = epi_warps_for(NT, MODE);
  static constexpr int THREADS = 96 + 32 * EPI_WARPS;
  static constexpr uint32_t ACC_COLS = NUM_A * NT;
  static constexpr int ACC_BUFS = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr uint32_t TMEM_COLS = pow2_at_least(ACC_BUFS * ACC_COLS);
  static constexpr uint32_t NUM_BARS = 2 * SA + 2 * SB + 2 * ACC_BUFS + 1;
  static constexpr uint32_t MISC_BYTES = 16 + 4 * (3 * kMaxE + 1);
  static constexpr uint32_t SMEM_BYTES =
      1024 + SA * A_STAGE + SB * B_STAGE + NUM_BARS * 8 + MISC_BYTES;
  static_assert(B_STAGE % 1024 == 0, "token tile must keep 1024-byte alignment");
  static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(SB >= 2, "token ring needs two stages");
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 256, "MMA N for M = 128");
};

__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

template <int NT, int MODE, bool F8>
__global__ void __launch_bounds__(threads_for(NT, MODE), 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0,
                       const __grid_constant__ CUtensorMap tm_a1,
                       const __grid_constant__ CUtensorMap tm_b, const GemmArgs p) {
  using C = Cfg<NT, MODE>;
  constexpr bool GATEUP = MODE == kModeGateUp;
  constexpr bool PAIR = MODE == kModeDownPair;
  // decode-sized token blocks gather their rows from the hidden states with
  // per-row TMA loads; larger blocks load whole tiles of a gathered copy
  constexpr bool ROW_GATHER = GATEUP && NT <= 32;
  constexpr int KE = F8 ? kRowBytes : kRowBytes / 2;  // K elements per K block
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t a_ring = raw_addr + pad;
  const uint32_t b_ring = a_ring + C::B_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::SA * C::A_STAGE + C::SB * C::B_STAGE);
  int32_t* misc = reinterpret_cast<int32_t*>(bars + C::NUM_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int32_t* abort_flag = misc + 1;
  int32_t* s_total = misc + 2;  // permuted rows of all experts (offsets[E])
  int32_t* s_cnt = misc + 4;
  int32_t* s_off = s_cnt + kMaxE;
  int32_t* s_start = s_off + kMaxE;

  const uint32_t bar0 = ptx::smem_addr(bars);
  auto fullA = [&](int s) { return bar0 + 8u * s; };
  auto emptyA = [&](int s) { return bar0 + 8u * (C::SA + s); };
  auto fullB = [&](int s) { return bar0 + 8u * (2 * C::SA + s); };
  auto emptyB = [&](int s) { return bar0 + 8u * (2 * C::SA + C::SB + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::SA + 2 * C::SB + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::SA + 2 * C::SB + C::ACC_BUFS + a); };
  const uint32_t done_bar = bar0 + 8u * (2 * C::SA + 2 * C::SB + 2 * C::ACC_BUFS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::SA; ++s) {
      ptx::mbar_init(fullA(s), 1);
      ptx::mbar_init(emptyA(s), 1);
    }
    for (int s = 0; s < C::SB; ++s) {
      ptx::mbar_init(fullB(s), 1);
      ptx::mbar_init(emptyB(s), 1);
    }
    for (int a = 0; a < C::ACC_BUFS; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 32 * C::EPI_WARPS);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
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
  // Launched behind the previous kernel (programmatic dependent launch).
  // gate/up's tile list comes from the permutation right before it, so it
  // waits here, then lets the down GEMM start: down CTAs take the SMs that
  // gate/up CTAs leave.  The down GEMM's list comes from that same
  // permutation, complete before gate/up let it start: it reads the list and
  // streams weights at once, and only its token producer waits (for h).
  if (GATEUP) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
  }
  if (threadIdx.x == 0) *s_total = p.offsets[E];
  for (int e = threadIdx.x; e < E; e += C::THREADS) {
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
  // a tile to work on: rows to process, and (debug build) every index of it
  // inside its buffers; every role decides alike, so a bad tile is skipped
  // by all of them
  auto use_tile = [&](const TileInfo& ti) {
    if (ti.nvalid <= 0) return false;
    return in_bounds(ti.expert >= 0 && ti.expert < E && ti.mblock >= 0 &&
                         ti.mblock < p.m_blocks && ti.row0 >= 0 &&
                         ti.row0 + ti.nvalid <= *s_total && ti.n_mma <= NT,
                     p.status);
  };

  if (warp == 0) {
    // ------------------------------------------------------ weight producer
    if (lane == 0) {
      const uint64_t pol_w =
          p.weight_evict_first ? ptx::policy_evict_first() : ptx::policy_evict_normal();
      int last_parity[C::SA];
#pragma unroll
      for (int s = 0; s < C::SA; ++s) last_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool withhold = p.withhold_first_load != 0 && blockIdx.x == 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
        if (!use_tile(ti)) continue;
        int a_row = ti.expert * p.rows_per_expert + ti.mblock * (PAIR ? 2 * BM : BM);
        // the box's rows inside the weight tensor (else read row 0: the stage
        // still fills and the tile's result is void)
        if (!in_bounds(a_row + (PAIR ? 2 * BM : BM) <= p.a_rows, p.status)) a_row = 0;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!W.wait(emptyA(stage), phase ^ 1u)) {
            ok = false;
            break;
          }
          if (withhold) {
            withhold = false;  // test aid: this stage never fills
          } else {
            const uint32_t st = a_ring + stage * C::A_STAGE;
            ptx::mbar_arrive_expect_tx(fullA(stage), C::A_STAGE);
            ptx::tma_load_2d(st, &tm_a0, fullA(stage), kb * KE, a_row, pol_w);
            if (GATEUP)
              ptx::tma_load_2d(st + C::A_BYTES, &tm_a1, fullA(stage), kb * KE, a_row, pol_w);
            if (PAIR)
              ptx::tma_load_2d(st + C::A_BYTES, &tm_a0, fullA(stage), kb * KE, a_row + BM, pol_w);
            last_parity[stage] = static_cast<int>(phase);
          }
          if (++stage == C::SA) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the CTA may not exit while a copy into its shared memory is in flight
#pragma unroll
      for (int s = 0; s < C::SA; ++s)
        if (last_parity[s] >= 0) W.wait_final(fullA(s), static_cast<uint32_t>(last_parity[s]));
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------- token producer
    // With ROW_GATHER every lane issues one 128-byte row load per token it
    // owns (box of one row; the row lands at its swizzled place in the tile);
    // otherwise lane 0 loads the whole token tile (x gathered into expert
    // order, or h).
    constexpr int RPL = (NT + 31) / 32;  // token rows per lane
    // h comes from the kernel before this one.  The combine after this
    // kernel is not let in early: tens of thousands of its blocks waiting on
    // the SMs slowed this GEMM at prefill sizes.
    if (!GATEUP) ptx::grid_dep_wait();
    const uint64_t pol_b = ptx::policy_evict_last();
    int last_parity[C::SB];
#pragma unroll
    for (int s = 0; s < C::SB; ++s) last_parity[s] = -1;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
      if (!use_tile(ti)) continue;
      int tok[RPL];
      if constexpr (ROW_GATHER) {
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
          const int r = lane + 32 * j;
          tok[j] = r < ti.nvalid ? p.perm_src[ti.row0 + r] / p.topk : -1;
          // a row of the hidden states (else row 0 is read into its place)
          if (r < ti.nvalid && !in_bounds(tok[j] >= 0 && tok[j] < p.b_rows, p.status)) tok[j] = 0;
        }
      }
      // (tile loads: the block's first row inside the gathered copy; a row
      // gather addresses the hidden states by token instead, checked above)
      const int b_row0 = ROW_GATHER || in_bounds(ti.row0 < p.b_rows, p.status) ? ti.row0 : 0;
      const uint32_t tx_bytes =
          ROW_GATHER ? static_cast<uint32_t>(ti.nvalid) * kRowBytes : C::B_STAGE;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        int okw = 1;
        if (lane == 0) okw = W.wait(emptyB(stage), phase ^ 1u) ? 1 : 0;
        okw = __shfl_sync(kFull, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        const uint32_t st = b_ring + stage * C::B_STAGE;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(fullB(stage), tx_bytes);
          if (!ROW_GATHER) ptx::tma_load_2d(st, &tm_b, fullB(stage), kb * KE, b_row0, pol_b);
        }
        if constexpr (ROW_GATHER) {
          __syncwarp();
#pragma unroll
          for (int j = 0; j < RPL; ++j)
            if (tok[j] >= 0)
              ptx::tma_load_2d(st + (lane + 32 * j) * kRowBytes, &tm_b, fullB(stage), kb * KE,
                               tok[j], pol_b);
        }
        last_parity[stage] = static_cast<int>(phase);
        if (++stage == C::SB) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < C::SB; ++s)
        if (last_parity[s] >= 0) W.wait_final(fullB(s), static_cast<uint32_t>(last_parity[s]));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_m = F8 ? ptx::idesc_e4m3_f32(BM, 0) : ptx::idesc_bf16_f32(BM, 0);
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
        if (!use_tile(ti)) continue;
        const uint32_t idesc = idesc_m | (static_cast<uint32_t>(ti.n_mma >> 3) << 17);
        if (!W.wait(tempty_bar(acc), acc_phase ^ 1u)) break;
        ptx::tc_fence_after();
        // the accumulators' TMEM columns inside the allocation
        in_bounds(acc * C::ACC_COLS + C::NUM_A * ti.n_mma <= C::TMEM_COLS, p.status);
        const uint32_t d0 = tmem_base + acc * C::ACC_COLS;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!W.wait(fullA(sa), pa) || !W.wait(fullB(sb), pb)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st = a_ring + sa * C::A_STAGE;
          const uint32_t bt = b_ring + sb * C::B_STAGE;
#pragma unroll
          for (int kk = 0; kk < kRowBytes / kMmaKBytes; ++kk) {
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            const uint32_t ko = kk * kMmaKBytes;
            const uint64_t bd = ptx::sdesc_sw128(bt + ko);
            if constexpr (F8) {
              ptx::mma_f8(d0, ptx::sdesc_sw128(st + ko), bd, idesc, accum);
              if (C::NUM_A == 2)
                ptx::mma_f8(d0 + NT, ptx::sdesc_sw128(st + C::A_BYTES + ko), bd, idesc, accum);
            } else {
              ptx::mma_bf16(d0, ptx::sdesc_sw128(st + ko), bd, idesc, accum);
              if (C::NUM_A == 2)
                ptx::mma_bf16(d0 + NT, ptx::sdesc_sw128(st + C::A_BYTES + ko), bd, idesc, accum);
            }
          }
          // free both stages once these MMAs have read them
          ptx::mma_commit(emptyA(sa));
          ptx::mma_commit(emptyB(sb));
          if (++sa == C::SA) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sb == C::SB) {
            sb = 0;
            pb ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(tfull_bar(acc));
        if (++acc == C::ACC_BUFS) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA this thread issued completes before TMEM is released
      ptx::mma_commit(done_bar);
      W.wait_final(done_bar, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int m = q * 32 + lane;
    // with more than 4 epilogue warps, warps 3-6 take the first columns,
    // warps 7-10 the next ones, and so on
    constexpr int COLS_PER_WARP = NT / (C::EPI_WARPS / 4);
    const int col_begin = ((warp - 3) >> 2) * COLS_PER_WARP;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile<NT>(tile, s_start, s_cnt, s_off, E);
      if (!use_tile(ti)) continue;
      if (!W.wait(tfull_bar(acc), acc_phase)) break;
      ptx::tc_fence_after();
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS;
      const int col = ti.mblock * BM + m;
      // E4M3 operands: the scales of this thread's weight row(s)
      float sw0 = 1.f, sw1 = 1.f;
      if constexpr (F8) {
        const int64_t wrow = static_cast<int64_t>(ti.expert) * p.rows_per_expert +
                             (PAIR ? ti.mblock * 2 * BM + m : col);
        sw0 = p.a0_scale[wrow];
        if constexpr (GATEUP) sw1 = p.a1_scale[wrow];
        if constexpr (PAIR) sw1 = p.a0_scale[wrow + BM];
      }
#pragma unroll 1
      for (int c0 = col_begin; c0 < min(ti.nvalid, col_begin + COLS_PER_WARP); c0 += 16) {
        // the chunk's TMEM columns inside its accumulator
        if (!in_bounds(c0 + 16 <= NT, p.status)) break;
        uint32_t ra[16];
        ptx::tmem_ld16(tq + c0, ra);
        // per-token factors of the chunk's 16 columns, one column per lane
        // (lanes 16-31 repeat 0-15), loaded while the TMEM load is in flight
        // and handed out by shuffles: gate/up's E4M3 token scale, or down's
        // routing weight (times the E4M3 row scale) and output row
        const int lrow = ti.row0 + c0 + (lane & 15);
        const bool lvalid = c0 + (lane & 15) < ti.nvalid;
        float lfac = 1.f;
        int lorow = lrow;
        if constexpr (GATEUP) {
          if constexpr (F8)
            if (lvalid) lfac = p.b_scale[p.perm_src[lrow] / p.topk];
        } else {
          if (lvalid) {
            lfac = F8 ? p.b_scale[lrow] * p.perm_w[lrow] : p.perm_w[lrow];
            if (p.out_rows) lorow = p.out_rows[lrow];
          }
        }
        if constexpr (GATEUP) {
          uint32_t rb[16];
          ptx::tmem_ld16(tq + NT + c0, rb);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            // c0 + j < ti.nvalid is the same on every lane of the warp
            if (c0 + j < ti.nvalid) {
              // (the same on every lane: the shuffle below needs all of them)
              const int64_t hrow = ti.row0 + c0 + j;
              if (!in_bounds(hrow < p.out_rows_cap && (ti.mblock + 1) * BM <= p.out_ld, p.status))
                continue;
              float g = __uint_as_float(ra[j]);
              float u = __uint_as_float(rb[j]);
              if constexpr (F8) {
                const float sx = __shfl_sync(kFull, lfac, j);
                g *= sw0 * sx;
                u *= sw1 * sx;
              }
              // fast exp and divide: relative error near 1e-6, far below the
              // BF16 rounding of h that follows
              const float h = __fdividef(g, 1.0f + __expf(-g)) * u;
              p.h_out[hrow * p.out_ld + col] = f32_to_bf16(h);
            }
          }
        } else if constexpr (PAIR) {
          uint32_t rb[16];
          ptx::tmem_ld16(tq + NT + c0, rb);
          ptx::tmem_wait_ld();
          // the pair's first 128 rows are output columns pcol, the next pcol + 128
          const int pcol = ti.mblock * 2 * BM + m;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {
              const float w = __shfl_sync(kFull, lfac, j);
              const int orow = __shfl_sync(kFull, lorow, j);
              if (!in_bounds(orow >= 0 && orow < p.out_rows_cap && pcol + BM < p.out_ld,
                             p.status))
                continue;
              float* dst = p.f32_out + static_cast<int64_t>(orow) * p.out_ld + pcol;
              // streaming stores: the FP32 rows are read once, by the
              // combine, and would otherwise push tiles out of L2
              __stcs(dst, F8 ? __uint_as_float(ra[j]) * sw0 * w : __uint_as_float(ra[j]) * w);
              __stcs(dst + BM, F8 ? __uint_as_float(rb[j]) * sw1 * w : __uint_as_float(rb[j]) * w);
            }
          }
        } else {
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {
              const float w = __shfl_sync(kFull, lfac, j);
              const int orow = __shfl_sync(kFull, lorow, j);
              if (!in_bounds(orow >= 0 && orow < p.out_rows_cap && col < p.out_ld, p.status))
                continue;
              __stcs(p.f32_out + static_cast<int64_t>(orow) * p.out_ld + col,
                     F8 ? __uint_as_float(ra[j]) * sw0 * w : __uint_as_float(ra[j]) * w);
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty_bar(acc));
      if (++acc == C::ACC_BUFS) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace
}  // namespace beam
