// FP32 router logits on the tensor cores for larger batches.
//
// The router is FP32: FP32 weights, accumulation and logits ("vLLM 实现
// Reflection Beam 501B MoE 模型 Day 0 支持", section "MoE and residual stream");
// SGLang computes it as a "BF16x3 GEMM" ("SGLang 原生支持 Reflection 的 Beam 并驱动
// 其生产 API", section "Highlights").  Here W_r = W_hi + W_mid + W_lo (three BF16
// planes, exact to 2^-24 relative) and x is BF16, so every product
// x * plane is exact in FP32.  What is not exact is the tensor core's own FP32
// accumulation, whose truncation error grows with the length of a chain of
// MMAs into one accumulator: chained over all of K it misses a 1e-5 relative
// bound.  So each 64-wide K block (four MMAs) accumulates into a fresh TMEM
// accumulator, and the epilogue warps add the blocks in FP32 registers, in
// K order (deterministic).
//
// Tile: 128 experts (MMA M) x up to 128 tokens (MMA N), A = planes [E, 3d]
// (per 64-wide K range: hi | mid | lo side by side), B = hidden rows [T, d].
// One pipeline stage holds a K range's three weight blocks and its token
// block, so each token block is loaded once for the three planes.  When the
// tiles do not fill the GPU, K is split over `ksplit` CTAs per tile: split c
// writes its partial logits to logits + c * T * E and the selection adds the
// partials in split order.
// Warp 0: TMA producer; warp 1: TMEM owner and MMA issuer; warps 2-17: four
// warps per TMEM lane quarter, each draining a quarter of the token columns.
// Waits are bounded as in the expert GEMMs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "launch_once.cuh"
#include "ptx.cuh"

namespace beam {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int PLANES = 3;         // hi, mid, lo: the three BF16 planes of W_r
constexpr int kSumGroup = 8;      // K ranges per first-level partial sum
constexpr int kEpiWarps = 16;
constexpr int kEpiCols = BN / (kEpiWarps / 4);
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = PLANES * A_BYTES + B_BYTES;  // one K range
constexpr int STAGES = 3;
constexpr uint32_t ACC_COLS = BN;
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
constexpr uint32_t NUM_BARS = 2 * STAGES + 4 + 1;
constexpr uint32_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;

struct Waiter {
  volatile int32_t* abort_flag;
  uint32_t* status;
  uint64_t limit_ns;
  __device__ bool wait(uint32_t bar, uint32_t parity) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if ((n & 63u) == 0) {
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > limit_ns) {
          *abort_flag = 1;
          latch_status(status, kStatusTimeout);
          return false;
        }
      }
    }
  }
  __device__ bool wait_final(uint32_t bar, uint32_t parity) const {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 0;; ++n) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if ((n & 63u) == 63u && ptx::globaltimer() - t0 > limit_ns) {
        latch_status(status, kStatusTimeout);
        return false;
      }
    }
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                     float* __restrict__ logits, int64_t T, int32_t E, int32_t d, int32_t ksplit,
                     uint32_t* status, uint64_t wait_limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t tiles = raw_addr + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  int32_t* misc = reinterpret_cast<int32_t*>(bars + NUM_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int32_t* abort_flag = misc + 1;

  const uint32_t bar0 = ptx::smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_blocks = E / BM;
  const int t_blocks = static_cast<int>((T + BN - 1) / BN);
  const int num_tiles = m_blocks * t_blocks;
  const int num_items = num_tiles * ksplit;  // (tile, K split)
  const int groups = d / BK;                 // K ranges
  // item -> tile, split and its K ranges [g0, g1); consecutive items share
  // the split (the same K range of W_r) and differ in the tile
  auto item_of = [&](int item, int& mb, int& tb, int& kc, int& g0, int& g1) {
    const int tile = item % num_tiles;
    kc = item / num_tiles;
    mb = tile % m_blocks;
    tb = tile / m_blocks;
    g0 = kc * groups / ksplit;
    g1 = (kc + 1) * groups / ksplit;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 32 * kEpiWarps);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_w);
    ptx::prefetch_tmap(&tm_x);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const Waiter W{abort_flag, status, wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_last();
      int last_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
        int mb, tb, kc, g0, g1;
        item_of(item, mb, tb, kc, g0, g1);
        for (int g = g0; g < g1; ++g) {
          if (!W.wait(empty_bar(stage), phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t st = tiles + stage * STAGE_BYTES;
          ptx::mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
#pragma unroll
          for (int pl = 0; pl < PLANES; ++pl)
            ptx::tma_load_2d(st + pl * A_BYTES, &tm_w, full_bar(stage), (PLANES * g + pl) * BK,
                             mb * BM, pol);
          ptx::tma_load_2d(st + PLANES * A_BYTES, &tm_x, full_bar(stage), g * BK, tb * BN, pol);
          last_parity[stage] = static_cast<int>(phase);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
#pragma unroll
      for (int s = 0; s < STAGES; ++s)
        if (last_parity[s] >= 0) W.wait_final(full_bar(s), static_cast<uint32_t>(last_parity[s]));
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
        int mb, tb, kc, g0, g1;
        item_of(item, mb, tb, kc, g0, g1);
        const int nvalid = static_cast<int>(T - static_cast<int64_t>(tb) * BN < BN ? T - static_cast<int64_t>(tb) * BN : BN);
        const uint32_t idesc = ptx::idesc_bf16_f32(BM, (nvalid + 15) & ~15);
        for (int g = g0; ok && g < g1; ++g) {
          // each K range into a fresh accumulator: its three planes, four
          // MMAs each, all reading the stage's one token block
          if (!W.wait(tempty_bar(acc), acc_phase ^ 1u) || !W.wait(full_bar(stage), phase)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d0 = tmem_base + acc * ACC_COLS;
          const uint32_t st = tiles + stage * STAGE_BYTES;
#pragma unroll
          for (int pl = 0; pl < PLANES; ++pl)
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              ptx::mma_bf16(d0, ptx::sdesc_sw128(st + pl * A_BYTES + kk * 32),
                            ptx::sdesc_sw128(st + PLANES * A_BYTES + kk * 32), idesc,
                            (pl | kk) ? 1u : 0u);
          ptx::mma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          ptx::mma_commit(tfull_bar(acc));
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      ptx::mma_commit(done_bar);
      W.wait_final(done_bar, 0);
    }
    __syncwarp();
  } else {
    const int ew = warp - 2;
    const int q = warp & 3;              // TMEM lane quarter
    const int part = ew >> 2;            // which kEpiCols token columns
    const int e_row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
      int mb, tb, kc, g0, g1;
      item_of(item, mb, tb, kc, g0, g1);
      const int nvalid = static_cast<int>(
          T - static_cast<int64_t>(tb) * BN < BN ? T - static_cast<int64_t>(tb) * BN : BN);
      float sum[kEpiCols], grp[kEpiCols];
#pragma unroll
      for (int i = 0; i < kEpiCols; ++i) sum[i] = grp[i] = 0.f;
      for (int g = 0; g < g1 - g0; ++g) {
        if (!W.wait(tfull_bar(acc), acc_phase)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tq =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_COLS + part * kEpiCols;
#pragma unroll
        for (int c = 0; c < kEpiCols / 16; ++c) {
          uint32_t r[16];
          ptx::tmem_ld16(tq + 16 * c, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) grp[16 * c + i] += __uint_as_float(r[i]);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(tempty_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        if ((g + 1) % kSumGroup == 0 || g + 1 == g1 - g0) {
#pragma unroll
          for (int i = 0; i < kEpiCols; ++i) {
            sum[i] += grp[i];
            grp[i] = 0.f;
          }
        }
      }
      if (!ok) break;
      const int e = mb * BM + e_row;
      float* out = logits + static_cast<int64_t>(kc) * T * E;
#pragma unroll
      for (int i = 0; i < kEpiCols; ++i) {
        const int col = part * kEpiCols + i;
        if (col < nvalid) out[(static_cast<int64_t>(tb) * BN + col) * E + e] = sum[i];
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

int router_tc_ksplit(int64_t T, int32_t E, int32_t d, int num_sms) {
  const int64_t tiles = static_cast<int64_t>(E / BM) * ((T + BN - 1) / BN);
  if (tiles <= 0) return 1;
  // as many splits as whole waves of (tile, split) items fill the SMs, at
  // most one per 8 K ranges and 16 in all
  int64_t ks = num_sms / tiles;
  const int64_t cap = std::min<int64_t>(16, std::max<int64_t>(1, (d / BK) / kSumGroup));
  return static_cast<int>(std::max<int64_t>(1, std::min(ks, cap)));
}

cudaError_t launch_router_tc(const CUtensorMap& w_planes, const CUtensorMap& x, float* logits,
                             int64_t T, int32_t E, int32_t d, int32_t ksplit, uint32_t* status,
                             uint64_t wait_limit_ns, int num_sms, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(E / BM) * ((T + BN - 1) / BN) * ksplit;
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  if (grid <= 0) return cudaSuccess;
  const cudaError_t err = smem_limit_once<router_tc_kernel>(SMEM_BYTES);
  if (err != cudaSuccess) return err;
  router_tc_kernel<<<grid, kThreads, SMEM_BYTES, s>>>(w_planes, x, logits, T, E, d, ksplit,
                                                      status, wait_limit_ns);
  return cudaGetLastError();
}

}  // namespace beam
