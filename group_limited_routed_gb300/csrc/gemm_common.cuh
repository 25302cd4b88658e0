// Pieces shared by the persistent grouped-GEMM kernels: bounded mbarrier
// waits and the on-device tile list (expert, weight block, token block).
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace beam {
namespace gemm {

struct Waiter {
  volatile int32_t* abort_flag;
  uint32_t* status;
  uint64_t limit_ns;

  // Wait for the phase of `parity`; false if another role aborted or the
  // wait ran out (then this CTA aborts and the status is latched).
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

  // Wait that ignores the abort flag (used to let issued work finish).
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

struct TileInfo {
  int expert, mblock, row0, nvalid, n_mma;
};

// Token blocks of one expert: ceil(cnt / NT) blocks of nearly equal size,
// each a multiple of 16 rows (the last one takes the remainder).
template <int NT>
__device__ __forceinline__ int token_blocks(int cnt) {
  return (cnt + NT - 1) / NT;
}

template <int NT>
__device__ __forceinline__ int block_rows(int cnt, int ntb) {
  const int per = (cnt + ntb - 1) / ntb;
  return min(NT, (per + 15) & ~15);
}

// tile index -> (expert, weight block, first permuted row, valid rows, MMA N)
template <int NT>
__device__ __forceinline__ TileInfo decode_tile(int tile, const int32_t* s_start,
                                                const int32_t* s_cnt, const int32_t* s_off,
                                                int E) {
  int lo = 0, hi = E;  // s_start[lo] <= tile < s_start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_start[mid] <= tile)
      lo = mid;
    else
      hi = mid;
  }
  const int local = tile - s_start[lo];
  const int cnt = s_cnt[lo];
  const int ntb = token_blocks<NT>(cnt);
  const int bs = block_rows<NT>(cnt, ntb);
  const int tb = local % ntb;
  TileInfo ti;
  ti.expert = lo;
  ti.mblock = local / ntb;
  ti.row0 = s_off[lo] + tb * bs;
  ti.nvalid = min(bs, cnt - tb * bs);
  ti.n_mma = (ti.nvalid + 15) & ~15;
  return ti;
}


}  // namespace gemm
}  // namespace beam
