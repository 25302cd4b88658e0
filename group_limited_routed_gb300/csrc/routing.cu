// Router, group-limited selection, permutation, gather and combine kernels.
//
// Router: logits = x W_r^T in FP32 ("vLLM 实现 Reflection Beam 501B MoE 模型
// Day 0 支持", section "MoE and residual stream": FP32 router weights,
// accumulation and logits).  Selection: sigmoid scores plus correction bias,
// best groups by the sum of their two best choice scores, top-k experts of
// the kept groups, weights renormalised over the sigmoid scores and scaled
// (same section; "SGLang 原生支持 Reflection 的 Beam 并驱动其生产 API", section
// "Dense Layers and Grouped MoE Routing").  Combine: FP32 sum of the weighted
// expert outputs in slot order, rounded once to BF16 (SGLang post, section
// "Fusion Optimizations": local expert summation, routed scaling, BF16
// rounding).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "common.cuh"
#include "launch_once.cuh"
#include "ptx.cuh"

namespace beam {
namespace {

namespace cg = cooperative_groups;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// ------------------------------------------------------------------ router
// Block: 32 tokens x 64 experts over one K range; 256 threads, each 4 tokens
// x 2 experts (a warp covers the 32 tokens and 8 experts, so a K step reads
// one 16-byte and one 8-byte shared-memory word per 8 FMAs), FP32 FMA in
// ascending K order, summed per 32-wide slice first (blocked summation keeps
// the rounding error of the 5120-term sum near 1e-7); fixed order =>
// deterministic.
constexpr int kRtTok = 32;
constexpr int kRtExp = 64;
constexpr int kRtK = 32;
constexpr int kRtDepth = 4;  // K slices whose loads are in flight together

__device__ __forceinline__ void router_tile(const RouterArgs& a, int bx, int by, int bz) {
  __shared__ __align__(16) float xs[kRtK][kRtTok + 4];
  __shared__ __align__(16) float ws[kRtK][kRtExp + 4];
  const int e0 = bx * kRtExp;
  const int64_t t0 = static_cast<int64_t>(by) * kRtTok;
  const int k_begin = bz * a.k_chunk;
  const int k_end = min(a.d, k_begin + a.k_chunk);
  const int tid = threadIdx.x;
  const int tg = tid & 7;                              // tokens 4 tg .. 4 tg + 3
  const int eg = ((tid & 31) >> 3) + 4 * (tid >> 5);   // experts 2 eg, 2 eg + 1
  float acc[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) acc[i][j] = 0.f;

  // the loads of up to four 32-wide K slices are issued together, so a
  // decode-sized K range (128) costs one memory round trip
  const int xr_row = tid >> 3, xr_col = (tid & 7) * 4;
  const bool x_ok = t0 + xr_row < a.T;
  const uint16_t* xsrc = a.x + (t0 + xr_row) * a.d + xr_col;
  uint2 xreg[kRtDepth];
  float4 wreg[kRtDepth][2];
  for (int kc0 = k_begin; kc0 < k_end; kc0 += kRtDepth * kRtK) {
#pragma unroll
    for (int q = 0; q < kRtDepth; ++q) {
      const int kc = kc0 + q * kRtK;
      xreg[q] = make_uint2(0u, 0u);
      wreg[q][0] = wreg[q][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kc < k_end) {
        if (x_ok) xreg[q] = *reinterpret_cast<const uint2*>(xsrc + kc);
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
          const int li = tid + rep * 256;
          const int r = li >> 3;
          const int c = (li & 7) * 4;
          if (e0 + r < a.E)
            wreg[q][rep] = *reinterpret_cast<const float4*>(a.w + static_cast<int64_t>(e0 + r) * a.d +
                                                            kc + c);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kRtDepth; ++q) {
      if (kc0 + q * kRtK >= k_end) break;
      xs[xr_col + 0][xr_row] = bf16_to_f32(static_cast<uint16_t>(xreg[q].x & 0xffffu));
      xs[xr_col + 1][xr_row] = bf16_to_f32(static_cast<uint16_t>(xreg[q].x >> 16));
      xs[xr_col + 2][xr_row] = bf16_to_f32(static_cast<uint16_t>(xreg[q].y & 0xffffu));
      xs[xr_col + 3][xr_row] = bf16_to_f32(static_cast<uint16_t>(xreg[q].y >> 16));
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int li = tid + rep * 256;
        const int r = li >> 3;
        const int c = (li & 7) * 4;
        ws[c + 0][r] = wreg[q][rep].x;
        ws[c + 1][r] = wreg[q][rep].y;
        ws[c + 2][r] = wreg[q][rep].z;
        ws[c + 3][r] = wreg[q][rep].w;
      }
      __syncthreads();
      // blocked summation: each 32-wide slice is summed on its own, then added
      float sl[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < kRtK; ++kk) {
        const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][tg * 4]);
        const float2 wv = *reinterpret_cast<const float2*>(&ws[kk][eg * 2]);
        const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sl[i][0] = fmaf(xa[i], wv.x, sl[i][0]);
          sl[i][1] = fmaf(xa[i], wv.y, sl[i][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) acc[i][j] += sl[i][j];
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t0 + tg * 4 + i;
    const int e = e0 + eg * 2;
    if (t < a.T && e < a.E) {
      float* dst = a.part + (static_cast<int64_t>(bz) * a.T + t) * a.E + e;
      *reinterpret_cast<float2*>(dst) = make_float2(acc[i][0], acc[i][1]);
    }
  }
}

// --------------------------------------------------------------- selection
// One token per block, thread e owns expert e (E <= 256 = blockDim).
//  1. logit: the router's split-K partials of expert e summed in split order;
//     score s = sigmoid(logit), choice score c = s + bias.
//  2. group score: top-1 + top-2 of c inside each group of S = E/G
//     consecutive experts (S a power of two <= 32, so a group is an aligned
//     segment of S lanes of one warp: a butterfly of log2(S) steps).
//  3. group g is kept when fewer than kg groups precede it in the order
//     (score desc, group asc).
//  4. expert e of a kept group takes slot r = the number of experts of kept
//     groups that precede it in the order (c desc, expert asc); r < k selects
//     it.  This ranking gives the same slots as k rounds of argmax.  Only the
//     top min(k, S) of each kept group (ranked inside the group by shuffles)
//     can take a slot, and every expert preceding one of the k selected is
//     itself selected, so ranking among those candidates gives the same
//     slots; they are packed into one array for vector loads.
//  5. weights: alpha * s / (sum of the k selected s in slot order), in FP64,
//     rounded once to FP32.
constexpr int kSelMaxG = 128;

__device__ __forceinline__ void select_token(const SelectArgs& a, int64_t t) {
  __shared__ float s_gs[kSelMaxG];
  __shared__ int s_pos[kSelMaxG];
  __shared__ __align__(16) float s_kc[256];
  __shared__ __align__(16) int s_ke[256];
  __shared__ int s_slot_e[32];
  __shared__ float s_slot_s[32];
  const int e = threadIdx.x;
  const int lane = e & 31;
  const int E = a.E;
  const int S = E / a.G;
  const bool live = e < E;
  const float bias = live ? a.bias[e] : 0.f;

  float lg = 0.f;
  if (live) {
    const float* src = a.part + t * E + e;
    const int64_t stride = a.T * E;
    lg = src[0];
    int sp = 1;
    for (; sp + 16 <= a.ksplit; sp += 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = src[(sp + u) * stride];
#pragma unroll
      for (int u = 0; u < 16; ++u) lg += v[u];
    }
    for (; sp < a.ksplit; ++sp) lg += src[sp * stride];
    if (a.logits) a.logits[t * E + e] = lg;
  }
  const float sc = live ? 1.0f / (1.0f + expf(-lg)) : 0.f;
  const float c = live ? sc + bias : -FLT_MAX;

  float m1 = c, m2 = -FLT_MAX;
  for (int o = S >> 1; o >= 1; o >>= 1) {
    const float b1 = __shfl_xor_sync(kFull, m1, o);
    const float b2 = __shfl_xor_sync(kFull, m2, o);
    const float n1 = fmaxf(m1, b1);
    const float n2 = fmaxf(fminf(m1, b1), fmaxf(m2, b2));
    m1 = n1;
    m2 = n2;
  }
  if (live && (lane & (S - 1)) == 0) s_gs[e / S] = m1 + m2;
  __syncthreads();
  // a kept group's place among the kept groups: its rank, below kg
  if (e < a.G) {
    const float v = s_gs[e];
    int before = 0;
    for (int h = 0; h < a.G; ++h) {
      const float u = s_gs[h];
      before += (u > v || (u == v && h < e)) ? 1 : 0;
    }
    s_pos[e] = before < a.kg ? before : -1;
  }
  __syncthreads();
  // expert rank inside its group, by shuffles over the group's S lanes
  const int pos = live ? s_pos[e / S] : -1;
  const int seg = lane & ~(S - 1);
  int lr = 0;
  for (int j = 0; j < S; ++j) {
    const float u = __shfl_sync(kFull, c, seg + j);
    lr += (u > c || (u == c && seg + j < lane)) ? 1 : 0;
  }
  // the top min(k, S) of each kept group are the only candidates for the k
  // slots, packed (any order: ties compare indices), padded to a multiple of
  // four with entries that precede nothing
  const int kk = a.k < S ? a.k : S;
  const int n = a.kg * kk;
  const int n4 = (n + 3) & ~3;
  const bool cand = pos >= 0 && lr < kk;
  if (cand) {
    s_kc[pos * kk + lr] = c;
    s_ke[pos * kk + lr] = e;
  }
  if (e >= n && e < n4) {
    s_kc[e] = -FLT_MAX;
    s_ke[e] = 1 << 30;
  }
  __syncthreads();
  if (cand) {
    int rank = 0;
    const float4* kc = reinterpret_cast<const float4*>(s_kc);
    const int4* ke = reinterpret_cast<const int4*>(s_ke);
#pragma unroll 4
    for (int i = 0; i < n4 / 4; ++i) {
      const float4 u = kc[i];
      const int4 f = ke[i];
      rank += (u.x > c || (u.x == c && f.x < e)) ? 1 : 0;
      rank += (u.y > c || (u.y == c && f.y < e)) ? 1 : 0;
      rank += (u.z > c || (u.z == c && f.z < e)) ? 1 : 0;
      rank += (u.w > c || (u.w == c && f.w < e)) ? 1 : 0;
    }
    if (rank < a.k) {
      s_slot_e[rank] = e;
      s_slot_s[rank] = sc;
    }
  }
  __syncthreads();
  if (e < a.k) {
    double ssum = 0.0;
    for (int r = 0; r < a.k; ++r) ssum += static_cast<double>(s_slot_s[r]);
    a.idx[t * a.k + e] = s_slot_e[e];
    a.w[t * a.k + e] =
        static_cast<float>(static_cast<double>(a.alpha) * static_cast<double>(s_slot_s[e]) / ssum);
  }
}

// ------------------------------------------------- selection, warp per token
// The same rule as select_token with one warp per token, for batches large
// enough that a block per token would run many waves of short blocks.  Lane
// l holds experts l, l + 32, ... (E % 32 == 0, so every lane is live).
//  1.-2. logits, scores and group scores exactly as in select_token (the
//     same FP32 operations in the same order; groups are aligned segments of
//     S lanes inside one row of 32 experts).
//  3. group g is kept when fewer than kg groups precede it (score desc,
//     group asc), ranked from the warp's copy of the group scores.
//  4. slot r takes the r-th expert of the kept groups in the order (c desc,
//     expert asc): k rounds of a warp argmax, the same slots as the ranking.
//  5. weights as in select_token: FP64 sum of the k scores in slot order.
constexpr int kSelWarps = 8;  // tokens per 256-thread block

__global__ void __launch_bounds__(32 * kSelWarps) select_warp_kernel(SelectArgs a) {
  __shared__ float s_gs[kSelWarps][kSelMaxG];
  __shared__ int s_keep[kSelWarps][kSelMaxG];
  __shared__ int s_slot_e[kSelWarps][32];
  __shared__ float s_slot_s[kSelWarps][32];
  const int wi = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kSelWarps + wi;
  if (t >= a.T) return;  // whole warps leave together
  const int E = a.E;
  const int J = E / 32;
  const int S = E / a.G;
  float sc[8], c[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sc[j] = 0.f;
    c[j] = -FLT_MAX;
    if (j < J) {
      const int e = 32 * j + lane;
      const float* src = a.part + t * E + e;
      const int64_t stride = a.T * E;
      float lg = src[0];
      for (int sp = 1; sp < a.ksplit; ++sp) lg += src[sp * stride];
      if (a.logits) a.logits[t * E + e] = lg;
      sc[j] = 1.0f / (1.0f + expf(-lg));
      c[j] = sc[j] + a.bias[e];
      // top-1 + top-2 of the S-lane segment (a group)
      float m1 = c[j], m2 = -FLT_MAX;
      for (int o = S >> 1; o >= 1; o >>= 1) {
        const float b1 = __shfl_xor_sync(kFull, m1, o);
        const float b2 = __shfl_xor_sync(kFull, m2, o);
        const float n1 = fmaxf(m1, b1);
        const float n2 = fmaxf(fminf(m1, b1), fmaxf(m2, b2));
        m1 = n1;
        m2 = n2;
      }
      if ((lane & (S - 1)) == 0) s_gs[wi][e / S] = m1 + m2;
    }
  }
  __syncwarp();
  for (int g = lane; g < a.G; g += 32) {
    const float v = s_gs[wi][g];
    int before = 0;
    for (int h = 0; h < a.G; ++h) {
      const float u = s_gs[wi][h];
      before += (u > v || (u == v && h < g)) ? 1 : 0;
    }
    s_keep[wi][g] = before < a.kg ? 1 : 0;
  }
  __syncwarp();
  // experts outside the kept groups never win a round
  unsigned live = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < J && s_keep[wi][(32 * j + lane) / S]) live |= 1u << j;
  for (int r = 0; r < a.k; ++r) {
    float bv = -FLT_MAX;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 32 * j + lane;
      if (((live >> j) & 1u) && (be == 0x7fffffff || c[j] > bv)) {
        bv = c[j];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oe = __shfl_xor_sync(kFull, be, o);
      if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    // be is the same on every lane: its owner records it and drops it
    if ((be & 31) == lane) {
      const int jw = be >> 5;
      float sw = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j == jw) sw = sc[j];
      live &= ~(1u << jw);
      s_slot_e[wi][r] = be;
      s_slot_s[wi][r] = sw;
    }
  }
  __syncwarp();
  if (lane < a.k) {
    double ssum = 0.0;
    for (int r = 0; r < a.k; ++r) ssum += static_cast<double>(s_slot_s[wi][r]);
    a.idx[t * a.k + lane] = s_slot_e[wi][lane];
    a.w[t * a.k + lane] = static_cast<float>(static_cast<double>(a.alpha) *
                                             static_cast<double>(s_slot_s[wi][lane]) / ssum);
  }
}

// ------------------------------------------------------------ router split
// planes[e] = for each 64-wide K range r: [hi | mid | lo] of that range, with
// hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid): each product with
// a BF16 x is exact in FP32, and hi + mid + lo equals w to within 2^-24
// relative.
// Four consecutive weights per thread (d % 64 == 0, so they share a 64-wide
// range): one 16-byte load, three 8-byte stores.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ w, int32_t E,
                                                           int32_t d, uint16_t* __restrict__ planes) {
  const int64_t n4 = static_cast<int64_t>(E) * d / 4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = (4 * i) / d, j = (4 * i) % d;
    const float4 v4 = reinterpret_cast<const float4*>(w)[i];
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    uint16_t p[3][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(v[q]);
      const float r1 = v[q] - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid);
      const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
      p[0][q] = *reinterpret_cast<const uint16_t*>(&hi);
      p[1][q] = *reinterpret_cast<const uint16_t*>(&mid);
      p[2][q] = *reinterpret_cast<const uint16_t*>(&lo);
    }
    uint16_t* blk = planes + e * 3 * d + (j / 64) * 192 + (j % 64);
#pragma unroll
    for (int pl = 0; pl < 3; ++pl)
      *reinterpret_cast<uint2*>(blk + 64 * pl) =
          make_uint2(p[pl][0] | (static_cast<uint32_t>(p[pl][1]) << 16),
                     p[pl][2] | (static_cast<uint32_t>(p[pl][3]) << 16));
  }
}

// ----------------------------------------------------------------- permute
// Block e: counts its rows, finds its first permuted row (entries with a
// smaller expert index) and writes its rows in (token, slot) order.  Each
// thread takes 8 consecutive entries per step; a block-wide exclusive scan of
// the per-thread match counts keeps the order stable.
constexpr int kPermPer = 8;

__device__ __forceinline__ void load8(const int32_t* __restrict__ idx, int64_t i0, int64_t n,
                                      int (&v)[kPermPer]) {
  if (i0 + kPermPer <= n) {
    const int4 a = *reinterpret_cast<const int4*>(idx + i0);
    const int4 b = *reinterpret_cast<const int4*>(idx + i0 + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < kPermPer; ++j) v[j] = i0 + j < n ? idx[i0 + j] : -1;
  }
}

__device__ __forceinline__ void permute_expert(const PermuteArgs& a, int e) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  __shared__ int s_cnt[8], s_below[8], s_warp[8];
  __shared__ int s_tot[2];
  constexpr int64_t kStep = 256 * kPermPer;

  // pass 1: this expert's entries and those of smaller experts; four steps'
  // loads are issued together (the pass is bound by load latency)
  constexpr int kAhead = 4;
  int cnt = 0, below = 0;
  for (int64_t base = 0; base < a.TK; base += kAhead * kStep) {
    int v[kAhead][kPermPer];
#pragma unroll
    for (int q = 0; q < kAhead; ++q) {
      const int64_t i0 = base + q * kStep + static_cast<int64_t>(tid) * kPermPer;
      if (i0 < a.TK) load8(a.idx, i0, a.TK, v[q]);
    }
#pragma unroll
    for (int q = 0; q < kAhead; ++q) {
      const int64_t i0 = base + q * kStep + static_cast<int64_t>(tid) * kPermPer;
      if (i0 >= a.TK) continue;
#pragma unroll
      for (int j = 0; j < kPermPer; ++j) {
        if (i0 + j >= a.TK) break;
        const int x = v[q][j] - a.id_base;
        if (static_cast<unsigned>(x) >= static_cast<unsigned>(a.E)) {
          if (e == 0) {
            a.pair_row[i0 + j] = -1;
            latch_status(a.status, kStatusDeviceCheck);
          }
          continue;
        }
        cnt += (x == e);
        below += (x < e);
      }
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    cnt += __shfl_xor_sync(kFull, cnt, o);
    below += __shfl_xor_sync(kFull, below, o);
  }
  if (lane == 0) {
    s_cnt[warp] = cnt;
    s_below[warp] = below;
  }
  __syncthreads();
  if (tid == 0) {
    int tc = 0, tb = 0;
    for (int w = 0; w < 8; ++w) {
      tc += s_cnt[w];
      tb += s_below[w];
    }
    s_tot[0] = tc;
    s_tot[1] = tb;
    a.counts[e] = tc;
    a.offsets[e] = tb;
    if (e == a.E - 1) a.offsets[a.E] = tb + tc;
  }
  __syncthreads();
  const int total = s_tot[0];
  const int first = s_tot[1];
  // pass 2: the entries in order; the next step's loads are issued before
  // this step's scan
  auto fetch = [&](int64_t i0, int (&v)[kPermPer]) {
    if (i0 < a.TK) {
      load8(a.idx, i0, a.TK, v);
#pragma unroll
      for (int j = 0; j < kPermPer; ++j) v[j] -= a.id_base;
    } else {
#pragma unroll
      for (int j = 0; j < kPermPer; ++j) v[j] = -1;
    }
  };
  int running = 0;
  int vn[kPermPer];
  fetch(static_cast<int64_t>(tid) * kPermPer, vn);
  for (int64_t base = 0; base < a.TK && running < total; base += kStep) {
    const int64_t i0 = base + static_cast<int64_t>(tid) * kPermPer;
    int v[kPermPer];
#pragma unroll
    for (int j = 0; j < kPermPer; ++j) v[j] = vn[j];
    fetch(i0 + kStep, vn);
    unsigned mask = 0;
#pragma unroll
    for (int j = 0; j < kPermPer; ++j) mask |= (v[j] == e ? 1u : 0u) << j;
    const int mine = __popc(mask);
    // exclusive scan of `mine` over the block (thread order = entry order)
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int woff = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int cw = s_warp[w];
      woff += (w < warp) ? cw : 0;
      tot += cw;
    }
    int row = first + running + woff + incl - mine;
#pragma unroll
    for (int j = 0; j < kPermPer; ++j) {
      if (mask & (1u << j)) {
        const int64_t i = i0 + j;
        // the permuted row inside [0, TK)
        if (in_bounds(row >= 0 && row < a.TK, a.status)) {
          a.perm_src[row] = static_cast<int>(i);
          a.pair_row[i] = row;
          a.perm_w[row] = a.w[i];
        }
        ++row;
      }
    }
    running += tot;
    __syncthreads();
  }
}

// ------------------------------------------------------ permute (large batches)
// The same stable (expert, token, slot) order as permute_expert, as a
// counting sort in one cooperative launch: (A) each block counts the experts
// of a chunk of entries; (B) block 0 turns the chunk counts into each chunk's
// first row per expert (per expert over chunks, then over experts); (C) each
// block writes its chunk in order, 256 entries at a time: warp match-any
// groups equal experts, their ranks by lane, per-warp counts in shared memory
// order the warps.  Needs E <= 256 and chunk counts [ceil(TK/kSortChunk), E].
constexpr int kSortChunk = 1024;

__global__ void __launch_bounds__(256) permute_sort_kernel(PermuteArgs a, int32_t* hist) {
  cg::grid_group grid = cg::this_grid();
  __shared__ int s_h[256];
  __shared__ int s_wc[8][256];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  const int nc = static_cast<int>((a.TK + kSortChunk - 1) / kSortChunk);
  for (int c = blockIdx.x; c < nc; c += gridDim.x) {  // (A)
    for (int e = tid; e < E; e += 256) s_h[e] = 0;
    __syncthreads();
    const int64_t end = min(a.TK, static_cast<int64_t>(c + 1) * kSortChunk);
    for (int64_t i = static_cast<int64_t>(c) * kSortChunk + tid; i < end; i += 256) {
      const int v = a.idx[i] - a.id_base;
      if (static_cast<unsigned>(v) < static_cast<unsigned>(E)) {
        atomicAdd(&s_h[v], 1);
      } else {
        a.pair_row[i] = -1;
        latch_status(a.status, kStatusDeviceCheck);
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += 256) hist[static_cast<int64_t>(c) * E + e] = s_h[e];
    __syncthreads();
  }
  grid.sync();
  if (blockIdx.x == 0) {  // (B)
    int tot = 0;
    if (tid < E) {
      int c = 0;
      for (; c + 8 <= nc; c += 8) {
        int h[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) h[u] = hist[static_cast<int64_t>(c + u) * E + tid];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          hist[static_cast<int64_t>(c + u) * E + tid] = tot;
          tot += h[u];
        }
      }
      for (; c < nc; ++c) {
        const int h = hist[static_cast<int64_t>(c) * E + tid];
        hist[static_cast<int64_t>(c) * E + tid] = tot;
        tot += h;
      }
    }
    // exclusive scan of the totals over experts, in expert order
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_wc[0][warp] = incl;
    __syncthreads();
    int woff = 0, all = 0;
    for (int w = 0; w < 8; ++w) {
      woff += w < warp ? s_wc[0][w] : 0;
      all += s_wc[0][w];
    }
    const int off = woff + incl - tot;
    if (tid < E) {
      a.counts[tid] = tot;
      a.offsets[tid] = off;
      for (int c = 0; c < nc; ++c) hist[static_cast<int64_t>(c) * E + tid] += off;
    }
    if (tid == 0) a.offsets[E] = all;
  }
  grid.sync();
  for (int e = tid; e < 256; e += 256)
    for (int w = 0; w < 8; ++w) s_wc[w][e] = 0;
  for (int c = blockIdx.x; c < nc; c += gridDim.x) {  // (C)
    __syncthreads();
    for (int e = tid; e < E; e += 256) s_h[e] = hist[static_cast<int64_t>(c) * E + e];
    __syncthreads();
    const int64_t end = min(a.TK, static_cast<int64_t>(c + 1) * kSortChunk);
    for (int64_t sb = static_cast<int64_t>(c) * kSortChunk; sb < end; sb += 256) {
      const int64_t i = sb + tid;
      const int v = i < end ? a.idx[i] - a.id_base : -1;
      const bool valid = static_cast<unsigned>(v) < static_cast<unsigned>(E);
      const unsigned peers = __match_any_sync(kFull, valid ? v : (0x40000000 | lane));
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (valid && rank == 0) s_wc[warp][v] = __popc(peers);
      __syncthreads();
      int before = 0, total = 0;
      if (valid) {
        for (int w = 0; w < 8; ++w) {
          const int x = s_wc[w][v];
          before += w < warp ? x : 0;
          total += x;
        }
        const int pos = s_h[v] + before + rank;
        // the permuted row inside [0, TK)
        if (in_bounds(pos >= 0 && pos < a.TK, a.status)) {
          a.perm_src[pos] = static_cast<int>(i);
          a.pair_row[i] = pos;
          a.perm_w[pos] = a.w[i];
        }
      }
      __syncthreads();
      if (valid && before + rank + 1 == total) s_h[v] += total;
      if (valid && rank == 0) s_wc[warp][v] = 0;
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------------ gather
// Block t: token t's row of x, read once, written to each of its k permuted
// rows pair_row[t * k + j] (x_perm in expert order for the larger token
// blocks); a slot whose pair_row is -1 (an out-of-range or foreign routed
// index) is skipped.  n16 16-bit words per row, a multiple of 8.
__global__ void __launch_bounds__(128) scatter_tokens_kernel(const uint16_t* __restrict__ x,
                                                             const int32_t* __restrict__ pair_row,
                                                             int32_t k, int32_t n16,
                                                             uint16_t* __restrict__ xp,
                                                             uint32_t* status) {
  const int64_t t = blockIdx.x;
  __shared__ int64_t s_row[32];
  if (threadIdx.x < k) {
    const int64_t row = pair_row[t * k + threadIdx.x];
    // a row of x_perm: fewer than T * k of them
    s_row[threadIdx.x] =
        in_bounds(row < static_cast<int64_t>(gridDim.x) * k, status) ? row : -1;
  }
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(x + t * n16);
  constexpr int U = 8;
  const int n8 = n16 / 8;
  for (int base = threadIdx.x; base < n8; base += U * blockDim.x) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + u * blockDim.x < n8) r[u] = src[base + u * blockDim.x];
    for (int j = 0; j < k; ++j) {
      if (s_row[j] < 0) continue;  // an invalid routed index has no permuted row
      uint4* dst = reinterpret_cast<uint4*>(xp + s_row[j] * n16);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (base + u * blockDim.x < n8) dst[base + u * blockDim.x] = r[u];
    }
  }
}

// x_perm[row] = x[token of row] for the larger token blocks; rows past the
// last valid one are skipped.
__global__ void __launch_bounds__(128) gather_kernel(const uint16_t* __restrict__ x,
                                                     const int32_t* __restrict__ perm_src,
                                                     const int32_t* __restrict__ n_valid,
                                                     int32_t k, int32_t d,
                                                     uint16_t* __restrict__ xp) {
  const int64_t row = blockIdx.x;
  if (row >= *n_valid) return;
  const int64_t t = perm_src[row] / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
  uint4* dst = reinterpret_cast<uint4*>(xp + row * d);
  // all of a thread's loads are issued before its stores
  constexpr int U = 8;
  const int n8 = d / 8;
  for (int base = threadIdx.x; base < n8; base += U * blockDim.x) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + u * blockDim.x < n8) r[u] = src[base + u * blockDim.x];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + u * blockDim.x < n8) dst[base + u * blockDim.x] = r[u];
  }
}

// ----------------------------------------------------------------- combine
// out[t] = bf16( sum over slots, in slot order, of y[row(t, slot)] ) in FP32.
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ y,
                                                      const int32_t* __restrict__ pair_row,
                                                      int32_t k, int32_t d,
                                                      uint16_t* __restrict__ out,
                                                      uint32_t* status) {
  ptx::grid_dep_wait();  // y comes from the kernel before this one
  const int64_t t = blockIdx.x;
  const int c8 = blockIdx.y * blockDim.x + threadIdx.x;
  if (c8 >= d / 8) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  // up to 8 slots at a time: their rows, then their loads, then the sums in
  // slot order
  constexpr int kAhead = 8;
  for (int s0 = 0; s0 < k; s0 += kAhead) {
    int row[kAhead];
#pragma unroll
    for (int j = 0; j < kAhead; ++j) {
      row[j] = s0 + j < k ? pair_row[t * k + s0 + j] : -1;
      // a row of y: fewer than T * k of them
      if (!in_bounds(row[j] < static_cast<int64_t>(gridDim.x) * k, status)) row[j] = -1;
    }
    float4 a[kAhead], b[kAhead];
#pragma unroll
    for (int j = 0; j < kAhead; ++j) {
      if (row[j] >= 0) {
        const float4* src =
            reinterpret_cast<const float4*>(y + static_cast<int64_t>(row[j]) * d) + 2 * c8;
        a[j] = src[0];
        b[j] = src[1];
      }
    }
#pragma unroll
    for (int j = 0; j < kAhead; ++j) {
      if (row[j] < 0) continue;
      acc[0] += a[j].x;
      acc[1] += a[j].y;
      acc[2] += a[j].z;
      acc[3] += a[j].w;
      acc[4] += b[j].x;
      acc[5] += b[j].y;
      acc[6] += b[j].z;
      acc[7] += b[j].w;
    }
  }
  uint4 o;
  uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    ow[i] = static_cast<uint32_t>(f32_to_bf16(acc[2 * i])) |
            (static_cast<uint32_t>(f32_to_bf16(acc[2 * i + 1])) << 16);
  reinterpret_cast<uint4*>(out + t * d)[c8] = o;
}

// -------------------------------------------------- combine + boundary
// One block per token, FP32 arithmetic, BF16 roundings where the decoder
// keeps them: the combine exactly as combine_kernel (written to out); the
// post-norm p = bf16(m * g_post / sqrt(mean(m^2) + eps)); the depth-scaled
// residual add h' = bf16(bf16(c_h * h) + bf16(c_x * p)) (written over the
// residual stream); the next pre-norm x = bf16(h' * g_pre / sqrt(mean(h'^2) +
// eps)).  Sums of squares: per thread in chunk order, then a fixed-order
// block reduction, so the result is deterministic.
__device__ __forceinline__ float bf16r(float v) { return bf16_to_f32(f32_to_bf16(v)); }

__device__ __forceinline__ float block_sum(float v, float* s_red) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();  // s_red may still be read from the previous reduction
  if ((threadIdx.x & 31) == 0) s_red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < nw; ++w) t += s_red[w];
  return t;
}

__global__ void __launch_bounds__(256) combine_boundary_kernel(const float* __restrict__ y,
                                                               const int32_t* __restrict__ pair_row,
                                                               int32_t k, int32_t d,
                                                               uint16_t* __restrict__ out,
                                                               BoundaryArgs b, uint32_t* status) {
  extern __shared__ float s_v[];  // [d] the token's current values
  __shared__ float s_red[32];
  ptx::grid_dep_wait();  // y comes from the kernel before this one
  const int64_t t = blockIdx.x;
  const int n8 = d / 8;
  float ss = 0.f;
  for (int c8 = threadIdx.x; c8 < n8; c8 += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int sl = 0; sl < k; ++sl) {
      const int row = pair_row[t * k + sl];
      if (row < 0 || !in_bounds(row < static_cast<int64_t>(gridDim.x) * k, status)) continue;
      const float4* src = reinterpret_cast<const float4*>(y + static_cast<int64_t>(row) * d) + 2 * c8;
      const float4 a = src[0];
      const float4 c = src[1];
      acc[0] += a.x;
      acc[1] += a.y;
      acc[2] += a.z;
      acc[3] += a.w;
      acc[4] += c.x;
      acc[5] += c.y;
      acc[6] += c.z;
      acc[7] += c.w;
    }
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = f32_to_bf16(acc[2 * i]), hi = f32_to_bf16(acc[2 * i + 1]);
      ow[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      const float vl = bf16_to_f32(lo), vh = bf16_to_f32(hi);
      s_v[c8 * 8 + 2 * i] = vl;
      s_v[c8 * 8 + 2 * i + 1] = vh;
      ss = fmaf(vl, vl, ss);
      ss = fmaf(vh, vh, ss);
    }
    reinterpret_cast<uint4*>(out + t * d)[c8] = o;
  }
  const float r = 1.0f / sqrtf(block_sum(ss, s_red) / static_cast<float>(d) + b.eps);
  float ss2 = 0.f;
  for (int c8 = threadIdx.x; c8 < n8; c8 += blockDim.x) {
    const uint4 hv = reinterpret_cast<const uint4*>(b.residual + t * d)[c8];
    const uint4 gv = reinterpret_cast<const uint4*>(b.g_post)[c8];
    const uint16_t* hs = reinterpret_cast<const uint16_t*>(&hv);
    const uint16_t* gs = reinterpret_cast<const uint16_t*>(&gv);
    uint4 o;
    uint16_t* os = reinterpret_cast<uint16_t*>(&o);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float p = bf16r(s_v[c8 * 8 + i] * r * bf16_to_f32(gs[i]));
      const float a = bf16r(b.c_h * bf16_to_f32(hs[i]));
      const uint16_t hn = f32_to_bf16(a + bf16r(b.c_x * p));
      os[i] = hn;
      const float v = bf16_to_f32(hn);
      s_v[c8 * 8 + i] = v;
      ss2 = fmaf(v, v, ss2);
    }
    reinterpret_cast<uint4*>(b.residual + t * d)[c8] = o;
  }
  const float r2 = 1.0f / sqrtf(block_sum(ss2, s_red) / static_cast<float>(d) + b.eps);
  for (int c8 = threadIdx.x; c8 < n8; c8 += blockDim.x) {
    const uint4 gv = reinterpret_cast<const uint4*>(b.g_pre)[c8];
    const uint16_t* gs = reinterpret_cast<const uint16_t*>(&gv);
    uint4 o;
    uint16_t* os = reinterpret_cast<uint16_t*>(&o);
#pragma unroll
    for (int i = 0; i < 8; ++i) os[i] = f32_to_bf16(s_v[c8 * 8 + i] * r2 * bf16_to_f32(gs[i]));
    reinterpret_cast<uint4*>(b.next_x + t * d)[c8] = o;
  }
}

// ------------------------------------------------------- expert-parallel pack
// Packed row r (expert order, hence grouped by owning rank) carries its
// expert and its routing weight; block 0 also counts the rows per owner.
__global__ void __launch_bounds__(256) ep_pack_kernel(const int32_t* __restrict__ idx,
                                                      const int32_t* __restrict__ perm_src,
                                                      const float* __restrict__ perm_w,
                                                      const int32_t* __restrict__ offsets,
                                                      int64_t TK, int32_t E, int32_t n_ranks,
                                                      int32_t* __restrict__ send_expert,
                                                      float* __restrict__ send_w,
                                                      int32_t* __restrict__ send_counts) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r < TK) {
    send_expert[r] = idx[perm_src[r]];
    send_w[r] = perm_w[r];
  }
  if (blockIdx.x == 0) {
    const int per = E / n_ranks;
    for (int q = threadIdx.x; q < n_ranks; q += blockDim.x)
      send_counts[q] = offsets[(q + 1) * per] - offsets[q * per];
  }
}

__global__ void __launch_bounds__(256) router_kernel(RouterArgs a) {
  router_tile(a, blockIdx.x, blockIdx.y, blockIdx.z);
}

__global__ void __launch_bounds__(256) select_kernel(SelectArgs a) { select_token(a, blockIdx.x); }

__global__ void __launch_bounds__(256) permute_kernel(PermuteArgs a) { permute_expert(a, blockIdx.x); }

// Router partials, selection and permutation in one cooperative launch (all
// blocks resident): grid-wide syncs separate the three steps, which removes
// two launches from a decode-sized call.
__global__ void __launch_bounds__(256) fused_route_kernel(RouterArgs ra, int ksplit, SelectArgs sa,
                                                          PermuteArgs pa) {
  cg::grid_group grid = cg::this_grid();
  const int nbx = (ra.E + kRtExp - 1) / kRtExp;
  const int nby = static_cast<int>((ra.T + kRtTok - 1) / kRtTok);
  const int tiles = nbx * nby * ksplit;
  // the block-wide syncs between iterations keep one item's shared-memory
  // reads ahead of the next item's writes
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    router_tile(ra, tile % nbx, (tile / nbx) % nby, tile / (nbx * nby));
    __syncthreads();
  }
  grid.sync();
  for (int64_t t = blockIdx.x; t < sa.T; t += gridDim.x) {
    select_token(sa, t);
    __syncthreads();
  }
  grid.sync();
  for (int e = blockIdx.x; e < pa.E; e += gridDim.x) {
    permute_expert(pa, e);
    __syncthreads();
  }
}

}  // namespace

void launch_router(const RouterArgs& a, int ksplit, cudaStream_t s) {
  dim3 grid((a.E + kRtExp - 1) / kRtExp, static_cast<unsigned>((a.T + kRtTok - 1) / kRtTok), ksplit);
  router_kernel<<<grid, 256, 0, s>>>(a);
}

void launch_select(const SelectArgs& a, cudaStream_t s) {
  // a block per token for small batches (more threads per token, one wave),
  // a warp per token from 256 tokens on
  if (a.T < 256) {
    select_kernel<<<static_cast<unsigned>(a.T), 256, 0, s>>>(a);
    return;
  }
  const int64_t blocks = (a.T + kSelWarps - 1) / kSelWarps;
  select_warp_kernel<<<static_cast<unsigned>(blocks), 32 * kSelWarps, 0, s>>>(a);
}

void launch_router_split(const float* w, int32_t E, int32_t d, uint16_t* planes, cudaStream_t s) {
  router_split_kernel<<<2 * 152, 256, 0, s>>>(w, E, d, planes);
}

cudaError_t launch_fused_route(const RouterArgs& ra, int ksplit, const SelectArgs& sa,
                               const PermuteArgs& pa, int num_sms, cudaStream_t s) {
  // all blocks of a cooperative launch are resident at once
  const int per_sm = blocks_per_sm_once<fused_route_kernel>(256);
  if (per_sm <= 0) return cudaErrorUnknown;
  const int64_t tiles = static_cast<int64_t>((ra.E + kRtExp - 1) / kRtExp) *
                        ((ra.T + kRtTok - 1) / kRtTok) * ksplit;
  int64_t want = tiles;
  if (sa.T > want) want = sa.T;
  if (pa.E > want) want = pa.E;
  const int64_t cap = static_cast<int64_t>(per_sm) * num_sms;
  const int grid = static_cast<int>(want < cap ? want : cap);
  RouterArgs a0 = ra;
  SelectArgs a1 = sa;
  PermuteArgs a2 = pa;
  void* args[] = {&a0, &ksplit, &a1, &a2};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(fused_route_kernel), dim3(grid),
                                     dim3(256), args, 0, s);
}

cudaError_t launch_combine_boundary(const float* y, const int32_t* pair_row, int64_t T, int32_t k,
                                    int32_t d, uint16_t* out, const BoundaryArgs& b,
                                    uint32_t* status, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(d) * sizeof(float);
  // the largest row the entry point accepts (d <= 51200)
  const cudaError_t e = smem_limit_once<combine_boundary_kernel>(200 * 1024);
  if (e != cudaSuccess) return e;
  return launch_dependent(combine_boundary_kernel, dim3(static_cast<unsigned>(T)), dim3(256), smem,
                          s, y, pair_row, k, d, out, b, status);
}

void launch_ep_pack(const int32_t* idx, const int32_t* perm_src, const float* perm_w,
                    const int32_t* offsets, int64_t TK, int32_t E, int32_t n_ranks,
                    int32_t* send_expert, float* send_w, int32_t* send_counts, cudaStream_t s) {
  const int64_t blocks = TK > 0 ? (TK + 255) / 256 : 1;
  ep_pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      idx, perm_src, perm_w, offsets, TK, E, n_ranks, send_expert, send_w, send_counts);
}

cudaError_t launch_permute_sort(const PermuteArgs& a, int32_t* hist, int num_sms, cudaStream_t s) {
  const int per_sm = blocks_per_sm_once<permute_sort_kernel>(256);
  if (per_sm <= 0) return cudaErrorUnknown;
  const int64_t nc = (a.TK + kSortChunk - 1) / kSortChunk;
  const int64_t cap = static_cast<int64_t>(per_sm) * num_sms;
  const int grid = static_cast<int>(nc < cap ? (nc > 0 ? nc : 1) : cap);
  PermuteArgs a0 = a;
  void* args[] = {&a0, &hist};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(permute_sort_kernel), dim3(grid),
                                     dim3(256), args, 0, s);
}

void launch_permute(const PermuteArgs& a, cudaStream_t s) {
  permute_kernel<<<a.E, 256, 0, s>>>(a);
}

void launch_gather(const uint16_t* x, const int32_t* perm_src, const int32_t* n_valid, int64_t TK,
                   int32_t k, int32_t d, uint16_t* x_perm, cudaStream_t s) {
  gather_kernel<<<static_cast<unsigned>(TK), 128, 0, s>>>(x, perm_src, n_valid, k, d, x_perm);
}

void launch_scatter_tokens(const uint16_t* x, const int32_t* pair_row, int64_t T, int32_t k,
                           int32_t n16, uint16_t* x_perm, uint32_t* status, cudaStream_t s) {
  if (T <= 0) return;
  scatter_tokens_kernel<<<static_cast<unsigned>(T), 128, 0, s>>>(x, pair_row, k, n16, x_perm,
                                                                 status);
}

void launch_combine(const float* y, const int32_t* pair_row, int64_t T, int32_t k, int32_t d,
                    uint16_t* out, uint32_t* status, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(T), (d / 8 + 127) / 128);
  launch_dependent(combine_kernel, grid, dim3(128), 0, s, y, pair_row, k, d, out, status);
}

}  // namespace beam
