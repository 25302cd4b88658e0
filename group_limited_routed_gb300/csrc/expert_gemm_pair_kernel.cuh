// Device code of the paired-CTA grouped expert GEMMs (launched from
// expert_gemm.cu, the one file that includes this header): the 256-token
// blocks of larger batches.
//
// The same two GEMMs as expert_gemm_kernel.cuh -- gate/up with the FP32
// SwiGLU epilogue, down with the FP32 routing weight -- on a cluster of two
// CTAs that run on an SM pair and share one tensor-core MMA of M = 256
// (tcgen05.mma.cta_group::2).  A pair tile is 256 weight rows of one expert
// (gate and up rows for gate/up, W_d rows for down) times one block of up to
// 256 of the expert's permuted token rows:
//
//   CTA r (r = 0, 1) stages weight rows [128 r, 128 r + 128) of the tile
//   and token rows [r N/2, r N/2 + N/2) of the block (N = the block's rows
//   rounded up to 16) in its own shared memory; the leader (r = 0) issues the
//   MMAs, which read A from both CTAs (128 rows each) and B from both (N/2
//   rows each); each CTA's TMEM receives its 128 weight rows x N columns,
//   and each CTA's epilogue drains its own.
//
// So each SM holds half of the token block instead of all of it: a gate/up
// stage is 32 KB of weights plus 16 KB of tokens (four stages in flight
// instead of three), for the same MMA work per SM and stage.  The down GEMM
// (kModeDownPair) takes 512 weight rows per tile as two 256-row
// accumulators, the same stage shape.  The template also covers one 256-row
// accumulator per tile (kModeDown: 16 + 16 KB stages, the accumulator fits
// twice in TMEM); the launcher does not instantiate it, as it measured
// slower on the Beam shapes, and shapes whose d is not a multiple of 512
// take the single-CTA kernels.
//
// Protocol (every wait bounded, as in the single-CTA kernel):
//   - TMEM is allocated and freed collectively by one warp of each CTA;
//   - both CTAs' producers load into their own shared memory and count the
//     bytes on the leader's full barriers (the leader arms each with both
//     CTAs' byte count);
//   - the leader's MMA commits arrive on both CTAs' empty barriers (each
//     producer waits on its own) and on both CTAs' accumulator barriers;
//   - each epilogue warp of either CTA arrives on the leader's
//     accumulator-free barrier once it has drained its columns;
//   - a cluster barrier after the set-up (barriers initialised, TMEM
//     allocated) and one before the teardown (no more cross-CTA signals or
//     reads) bracket the work; every path of every role reaches both.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "expert_gemm.cuh"
#include "expert_gemm_kernel.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace beam {
namespace {

constexpr int kPairNT = 256;     // token rows of a pair tile's block
constexpr int kPairHalf = 128;   // token rows each CTA stages (the TMA box)
constexpr int kPairEpiWarps = 16;
constexpr uint64_t kPeerDrainNs = 1000000ull;  // see the producers' teardown

template <int MODE>
struct PairCfg {
  static constexpr bool GATEUP = MODE == kModeGateUp;
  // gate/up: the gate and up rows; down pair: two 256-row W_d blocks (each
  // split over the two CTAs), sharing the token operand
  static constexpr int NUM_A = MODE == kModeDown ? 1 : 2;
  static constexpr uint32_t A_BYTES = BM * kRowBytes;         // 128 weight rows
  static constexpr uint32_t A_STAGE = NUM_A * A_BYTES;
  static constexpr uint32_t B_STAGE = kPairHalf * kRowBytes;  // 128 token rows
  static constexpr int S_RAW = static_cast<int>(kTileBudget / (A_STAGE + B_STAGE));
  static constexpr int S = S_RAW > 8 ? 8 : S_RAW;
  static constexpr uint32_t B_RING = S * A_STAGE;              // offset of the token ring
  static constexpr int EPI_WARPS = kPairEpiWarps;
  static constexpr int THREADS = 96 + 32 * EPI_WARPS;
  static constexpr uint32_t ACC_COLS = NUM_A * kPairNT;
  static constexpr int ACC_BUFS = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr uint32_t TMEM_COLS = ACC_BUFS * ACC_COLS;
  static constexpr uint32_t NUM_BARS = 4 * S + 2 * ACC_BUFS + 1;
  static constexpr uint32_t MISC_BYTES = 16 + 4 * (3 * kMaxE + 1);
  static constexpr uint32_t SMEM_BYTES =
      1024 + S * (A_STAGE + B_STAGE) + NUM_BARS * 8 + MISC_BYTES;
  static_assert(B_STAGE % 1024 == 0 && A_STAGE % 1024 == 0, "1024-byte stage alignment");
  static_assert(TMEM_COLS == 512, "TMEM has 512 columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(S >= 3, "ring depth");
};

template <int MODE, bool F8>
__global__ void __launch_bounds__(PairCfg<MODE>::THREADS, 1)
    expert_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a0,
                            const __grid_constant__ CUtensorMap tm_a1,
                            const __grid_constant__ CUtensorMap tm_b, const GemmArgs p) {
  using C = PairCfg<MODE>;
  constexpr bool GATEUP = C::GATEUP;
  constexpr bool PAIR = MODE == kModeDownPair;
  // weight rows one tile covers: 256 per accumulator (128 in each CTA)
  constexpr int TILE_ROWS = (PAIR ? 2 : 1) * 2 * BM;
  constexpr int KE = F8 ? kRowBytes : kRowBytes / 2;  // K elements per K block
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t a_ring = raw_addr + pad;
  const uint32_t b_ring = a_ring + C::B_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::S * (C::A_STAGE + C::B_STAGE));
  int32_t* misc = reinterpret_cast<int32_t*>(bars + C::NUM_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int32_t* abort_flag = misc + 1;
  int32_t* s_total = misc + 2;  // permuted rows of all experts (offsets[E])
  int32_t* s_cnt = misc + 4;
  int32_t* s_off = s_cnt + kMaxE;
  int32_t* s_start = s_off + kMaxE;

  const uint32_t bar0 = ptx::smem_addr(bars);
  auto fullA = [&](int s) { return bar0 + 8u * s; };
  auto emptyA = [&](int s) { return bar0 + 8u * (C::S + s); };
  auto fullB = [&](int s) { return bar0 + 8u * (2 * C::S + s); };
  auto emptyB = [&](int s) { return bar0 + 8u * (3 * C::S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (4 * C::S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (4 * C::S + C::ACC_BUFS + a); };
  const uint32_t done_bar = bar0 + 8u * (4 * C::S + 2 * C::ACC_BUFS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;
  const uint32_t rank = ptx::cluster_rank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S; ++s) {
      ptx::mbar_init(fullA(s), 1);  // the leader's producer; bytes of both CTAs
      ptx::mbar_init(emptyA(s), 1);
      ptx::mbar_init(fullB(s), 1);
      ptx::mbar_init(emptyB(s), 1);
    }
    for (int a = 0; a < C::ACC_BUFS; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 2 * C::EPI_WARPS);  // every epilogue warp of both CTAs
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
    ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  // programmatic dependent launch, as in the single-CTA kernel: gate/up
  // waits for the permutation here; the down GEMM reads its tile list at
  // once and only its token producer waits (for h)
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
      const int v = e < E ? p.m_blocks * token_blocks<kPairNT>(s_cnt[e]) : 0;
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
  // both CTAs' barriers are initialised and the pair's TMEM allocated before
  // any signal crosses between them
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = s_start[E];
  const Waiter W{abort_flag, p.status, p.wait_limit_ns};
  auto use_tile = [&](const TileInfo& ti) {
    if (ti.nvalid <= 0) return false;
    return in_bounds(ti.expert >= 0 && ti.expert < E && ti.mblock >= 0 &&
                         ti.mblock < p.m_blocks && ti.row0 >= 0 &&
                         ti.row0 + ti.nvalid <= *s_total && ti.n_mma <= kPairNT,
                     p.status);
  };

  if (warp == 0 || warp == 2) {
    // ------------------------------------------- producers (weights, tokens)
    // Each CTA loads its own half of every stage into its own shared memory;
    // the bytes count on the leader's full barriers, which the leader's
    // producer arms with both halves' byte count.
    if (lane == 0) {
      const bool weights = warp == 0;
      if (!GATEUP && !weights) ptx::grid_dep_wait();  // h: the kernel before this one
      const uint32_t stage_bytes = weights ? C::A_STAGE : C::B_STAGE;
      const uint32_t ring = weights ? a_ring : b_ring;
      const uint64_t pol = weights ? (p.weight_evict_first ? ptx::policy_evict_first()
                                                           : ptx::policy_evict_normal())
                                   : ptx::policy_evict_last();
      int last_parity[C::S];
#pragma unroll
      for (int s = 0; s < C::S; ++s) last_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      uint64_t last_issue = 0;
      bool withhold = weights && leader && p.withhold_first_load != 0 && blockIdx.x == 0;
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        const TileInfo ti = decode_tile<kPairNT>(tile, s_start, s_cnt, s_off, E);
        if (!use_tile(ti)) continue;
        int row;
        if (weights) {
          row = ti.expert * p.rows_per_expert + ti.mblock * TILE_ROWS + static_cast<int>(rank) * BM;
          if (!in_bounds(row + (PAIR ? 2 * BM : 0) + BM <= p.a_rows, p.status)) row = 0;
        } else {
          // this CTA's half of the block: rows [r N/2, r N/2 + N/2); a half
          // with no valid row (a block of at most N/2 rows) may start at the
          // operand's end: its load is padding (zero fill), never read
          const int first = static_cast<int>(rank) * (ti.n_mma / 2);
          row = ti.row0 + first;
          if (!in_bounds(first >= ti.nvalid || row < p.b_rows, p.status)) row = 0;
        }
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          const uint32_t empty = weights ? emptyA(stage) : emptyB(stage);
          const uint32_t full = weights ? fullA(stage) : fullB(stage);
          if (!W.wait(empty, phase ^ 1u)) {
            ok = false;
            break;
          }
          if (leader) ptx::mbar_arrive_expect_tx(full, 2 * stage_bytes);
          const uint32_t lead_full = ptx::map_to_rank(full, 0);
          const uint32_t st = ring + stage * stage_bytes;
          if (withhold) {
            withhold = false;  // test aid: this stage never fills
          } else if (weights) {
            ptx::tma_load_2d_pair(st, &tm_a0, lead_full, kb * KE, row, pol);
            if (GATEUP) ptx::tma_load_2d_pair(st + C::A_BYTES, &tm_a1, lead_full, kb * KE, row, pol);
            // the second W_d block: rows 256 further (this CTA's half of it)
            if (PAIR)
              ptx::tma_load_2d_pair(st + C::A_BYTES, &tm_a0, lead_full, kb * KE, row + 2 * BM, pol);
          } else {
            ptx::tma_load_2d_pair(st, &tm_b, lead_full, kb * KE, row, pol);
          }
          last_issue = ptx::globaltimer();
          last_parity[stage] = static_cast<int>(phase);
          if (++stage == C::S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // The CTA may not exit while a copy into its shared memory is in
      // flight.  The leader's full barriers count both CTAs' bytes: once
      // the leader has seen its last phases complete, the peer's copies of
      // those phases have landed as well, and the cluster barrier below
      // keeps the peer until then.  After an abort the peer may have issued
      // copies for phases the leader never armed; it lets them land (a
      // 16 KB copy takes microseconds) before going on.
      if (leader) {
#pragma unroll
        for (int s = 0; s < C::S; ++s)
          if (last_parity[s] >= 0)
            W.wait_final(weights ? fullA(s) : fullB(s), static_cast<uint32_t>(last_parity[s]));
      } else if (!ok || *abort_flag) {
        while (ptx::globaltimer() - last_issue < kPeerDrainNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc_m =
          F8 ? ptx::idesc_e4m3_f32(2 * BM, 0) : ptx::idesc_bf16_f32(2 * BM, 0);
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        const TileInfo ti = decode_tile<kPairNT>(tile, s_start, s_cnt, s_off, E);
        if (!use_tile(ti)) continue;
        const uint32_t idesc = idesc_m | (static_cast<uint32_t>(ti.n_mma >> 3) << 17);
        if (!W.wait(tempty_bar(acc), acc_phase ^ 1u)) break;
        ptx::tc_fence_after();
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
              ptx::mma_f8_pair(d0, ptx::sdesc_sw128(st + ko), bd, idesc, accum);
              if (C::NUM_A == 2)
                ptx::mma_f8_pair(d0 + kPairNT, ptx::sdesc_sw128(st + C::A_BYTES + ko), bd, idesc,
                                 accum);
            } else {
              ptx::mma_bf16_pair(d0, ptx::sdesc_sw128(st + ko), bd, idesc, accum);
              if (C::NUM_A == 2)
                ptx::mma_bf16_pair(d0 + kPairNT, ptx::sdesc_sw128(st + C::A_BYTES + ko), bd, idesc,
                                   accum);
            }
          }
          // both CTAs' stages are free once these MMAs have read them
          ptx::mma_commit_pair_both(emptyA(sa));
          ptx::mma_commit_pair_both(emptyB(sb));
          if (++sa == C::S) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sb == C::S) {
            sb = 0;
            pb ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_both(tfull_bar(acc));
        if (++acc == C::ACC_BUFS) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued completes before TMEM is released
      ptx::mma_commit_pair_self(done_bar);
      W.wait_final(done_bar, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Each CTA drains its own 128 weight rows (its TMEM lanes) for every
    // column (token) of the tile, then one lane per warp frees the columns
    // on the leader's barrier.
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int m = q * 32 + lane;
    constexpr int COLS_PER_WARP = kPairNT / (C::EPI_WARPS / 4);
    const int col_begin = ((warp - 3) >> 2) * COLS_PER_WARP;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs) {
      const TileInfo ti = decode_tile<kPairNT>(tile, s_start, s_cnt, s_off, E);
      if (!use_tile(ti)) continue;
      if (!W.wait(tfull_bar(acc), acc_phase)) break;
      ptx::tc_fence_after();
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS;
      // this CTA's weight row: output column (h's f, or y's column; the
      // down pair's second accumulator is 256 columns further)
      const int col = ti.mblock * TILE_ROWS + static_cast<int>(rank) * BM + m;
      float sw0 = 1.f, sw1 = 1.f;
      if constexpr (F8) {
        const int64_t wrow = static_cast<int64_t>(ti.expert) * p.rows_per_expert + col;
        sw0 = p.a0_scale[wrow];
        if constexpr (GATEUP) sw1 = p.a1_scale[wrow];
        if constexpr (PAIR) sw1 = p.a0_scale[wrow + 2 * BM];
      }
      if constexpr (GATEUP) {
        // h of this lane's weight row for the warp's 64 tokens, kept in
        // registers as BF16 pairs: the accumulator is freed as soon as it
        // has been read, before any store, so the next tile's MMAs do not
        // wait for the h stores
        uint32_t hp[COLS_PER_WARP / 2];
#pragma unroll
        for (int cc = 0; cc < COLS_PER_WARP; cc += 16) {
          const int c0 = col_begin + cc;
          if (c0 >= ti.nvalid) break;  // the same on every lane of the warp
          uint32_t ra[16], rb[16];
          ptx::tmem_ld16(tq + c0, ra);
          ptx::tmem_ld16(tq + kPairNT + c0, rb);
          // per-token factors of the chunk's 16 columns, one column per
          // lane, handed out by shuffles (as in the single-CTA kernel)
          float lfac = 1.f;
          if constexpr (F8)
            if (c0 + (lane & 15) < ti.nvalid) lfac = p.b_scale[p.perm_src[ti.row0 + c0 + (lane & 15)] / p.topk];
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float hv[2];
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2) {
              float g = __uint_as_float(ra[j + u2]);
              float u = __uint_as_float(rb[j + u2]);
              if constexpr (F8) {
                const float sx = __shfl_sync(kFull, lfac, j + u2);
                g *= sw0 * sx;
                u *= sw1 * sx;
              }
              // fast exp and divide, as in the single-CTA kernel
              hv[u2] = __fdividef(g, 1.0f + __expf(-g)) * u;
            }
            hp[(cc + j) / 2] = static_cast<uint32_t>(f32_to_bf16(hv[0])) |
                               (static_cast<uint32_t>(f32_to_bf16(hv[1])) << 16);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ptx::map_to_rank(tempty_bar(acc), 0));
#pragma unroll
        for (int cc = 0; cc < COLS_PER_WARP; cc += 16) {
          const int c0 = col_begin + cc;
          if (c0 >= ti.nvalid) break;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {  // the same on every lane of the warp
              const int64_t hrow = ti.row0 + c0 + j;
              if (!in_bounds(hrow < p.out_rows_cap && (ti.mblock + 1) * TILE_ROWS <= p.out_ld,
                             p.status))
                continue;
              p.h_out[hrow * p.out_ld + col] =
                  static_cast<uint16_t>(hp[(cc + j) / 2] >> (16 * ((cc + j) & 1)));
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c0 = col_begin; c0 < min(ti.nvalid, col_begin + COLS_PER_WARP); c0 += 16) {
          if (!in_bounds(c0 + 16 <= kPairNT, p.status)) break;
          uint32_t ra[16];
          ptx::tmem_ld16(tq + c0, ra);
          // per-token factors of the chunk's 16 columns, one column per lane,
          // handed out by shuffles (as in the single-CTA kernel)
          const int lrow = ti.row0 + c0 + (lane & 15);
          const bool lvalid = c0 + (lane & 15) < ti.nvalid;
          float lfac = 1.f;
          int lorow = lrow;
          if (lvalid) {
            lfac = F8 ? p.b_scale[lrow] * p.perm_w[lrow] : p.perm_w[lrow];
            if (p.out_rows) lorow = p.out_rows[lrow];
          }
          uint32_t rb[16];
          if constexpr (PAIR) ptx::tmem_ld16(tq + kPairNT + c0, rb);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.nvalid) {
              const float w = __shfl_sync(kFull, lfac, j);
              const int orow = __shfl_sync(kFull, lorow, j);
              if (!in_bounds(orow >= 0 && orow < p.out_rows_cap &&
                                 col + (PAIR ? 2 * BM : 0) < p.out_ld,
                             p.status))
                continue;
              float* dst = p.f32_out + static_cast<int64_t>(orow) * p.out_ld + col;
              // streaming stores: the FP32 rows are read once, by the combine
              __stcs(dst, F8 ? __uint_as_float(ra[j]) * sw0 * w : __uint_as_float(ra[j]) * w);
              if constexpr (PAIR)
                __stcs(dst + 2 * BM,
                       F8 ? __uint_as_float(rb[j]) * sw1 * w : __uint_as_float(rb[j]) * w);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ptx::map_to_rank(tempty_bar(acc), 0));
      }
      if (++acc == C::ACC_BUFS) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // no signal, copy or MMA read crosses between the two CTAs after this
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace
}  // namespace beam
