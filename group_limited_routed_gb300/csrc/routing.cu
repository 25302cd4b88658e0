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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "common.cuh"

namespace beam {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// ------------------------------------------------------------------ router
// Block: 32 tokens x 64 experts over one K range; 256 threads, each 2 tokens
// x 4 experts, FP32 FMA in ascending K order, summed per 32-wide slice first
// (blocked summation keeps the rounding error of the 5120-term sum near
// 1e-7); fixed order => deterministic.
constexpr int kRtTok = 32;
constexpr int kRtExp = 64;
constexpr int kRtK = 32;

__global__ void __launch_bounds__(256) router_kernel(RouterArgs a) {
  __shared__ float xs[kRtK][kRtTok + 1];
  __shared__ __align__(16) float ws[kRtK][kRtExp + 4];
  const int e0 = blockIdx.x * kRtExp;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kRtTok;
  const int k_begin = blockIdx.z * a.k_chunk;
  const int k_end = min(a.d, k_begin + a.k_chunk);
  const int tid = threadIdx.x;
  const int tx = tid & 15;
  const int ty = tid >> 4;
  float acc[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  // register prefetch of the next 32-wide K slice overlaps its load latency
  // with the FMAs of the current one
  const int xr_row = tid >> 3, xr_col = (tid & 7) * 4;
  const bool x_ok = t0 + xr_row < a.T;
  const uint16_t* xsrc = a.x + (t0 + xr_row) * a.d + xr_col;
  uint2 xreg = make_uint2(0u, 0u);
  float4 wreg[2];
  auto load_slice = [&](int kc) {
    if (x_ok) xreg = *reinterpret_cast<const uint2*>(xsrc + kc);
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int li = tid + rep * 256;
      const int r = li >> 3;
      const int c = (li & 7) * 4;
      wreg[rep] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + r < a.E)
        wreg[rep] =
            *reinterpret_cast<const float4*>(a.w + static_cast<int64_t>(e0 + r) * a.d + kc + c);
    }
  };
  if (k_begin < k_end) load_slice(k_begin);
  for (int kc = k_begin; kc < k_end; kc += kRtK) {
    xs[xr_col + 0][xr_row] = bf16_to_f32(static_cast<uint16_t>(xreg.x & 0xffffu));
    xs[xr_col + 1][xr_row] = bf16_to_f32(static_cast<uint16_t>(xreg.x >> 16));
    xs[xr_col + 2][xr_row] = bf16_to_f32(static_cast<uint16_t>(xreg.y & 0xffffu));
    xs[xr_col + 3][xr_row] = bf16_to_f32(static_cast<uint16_t>(xreg.y >> 16));
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int li = tid + rep * 256;
      const int r = li >> 3;
      const int c = (li & 7) * 4;
      ws[c + 0][r] = wreg[rep].x;
      ws[c + 1][r] = wreg[rep].y;
      ws[c + 2][r] = wreg[rep].z;
      ws[c + 3][r] = wreg[rep].w;
    }
    __syncthreads();
    if (kc + kRtK < k_end) load_slice(kc + kRtK);
    // blocked summation: each 32-wide slice is summed on its own, then added
    float sl[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < kRtK; ++kk) {
      const float x0 = xs[kk][ty * 2];
      const float x1 = xs[kk][ty * 2 + 1];
      const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      sl[0][0] = fmaf(x0, wv.x, sl[0][0]);
      sl[0][1] = fmaf(x0, wv.y, sl[0][1]);
      sl[0][2] = fmaf(x0, wv.z, sl[0][2]);
      sl[0][3] = fmaf(x0, wv.w, sl[0][3]);
      sl[1][0] = fmaf(x1, wv.x, sl[1][0]);
      sl[1][1] = fmaf(x1, wv.y, sl[1][1]);
      sl[1][2] = fmaf(x1, wv.z, sl[1][2]);
      sl[1][3] = fmaf(x1, wv.w, sl[1][3]);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] += sl[i][j];
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t t = t0 + ty * 2 + i;
    const int e = e0 + tx * 4;
    if (t < a.T && e < a.E) {
      float* dst = a.part + (static_cast<int64_t>(blockIdx.z) * a.T + t) * a.E + e;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
  }
}

// --------------------------------------------------------------- selection
// Phase 1 (whole block): thread e sums the router's split-K partials of
// expert e for each token of the block, in split order, into shared memory.
// Phase 2: one warp per token.  Lane l holds experts j*32 + l (j < E/32).
// Groups are S = E/G consecutive experts, S a power of two <= 32, so a group
// is an aligned segment of S lanes of one register.
constexpr int kSelMaxTok = 8;

__global__ void __launch_bounds__(256) select_kernel(SelectArgs a, int tok_per_block) {
  __shared__ float s_logit[kSelMaxTok][256];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tok_per_block;
  const int E = a.E;
  for (int tk = 0; tk < tok_per_block; ++tk) {
    const int64_t t = t0 + tk;
    const int e = threadIdx.x;
    if (t < a.T && e < E) {
      const float* src = a.part + t * E + e;
      const int64_t stride = a.T * E;
      float lg = src[0];
      int sp = 1;
      for (; sp + 8 <= a.ksplit; sp += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = src[(sp + u) * stride];
#pragma unroll
        for (int u = 0; u < 8; ++u) lg += v[u];
      }
      for (; sp < a.ksplit; ++sp) lg += src[sp * stride];
      s_logit[tk][e] = lg;
      if (a.logits) a.logits[t * E + e] = lg;
    }
  }
  __syncthreads();
  if (warp >= tok_per_block) return;
  const int64_t t = t0 + warp;
  if (t >= a.T) return;
  const int epl = E >> 5;
  const int S = E / a.G;

  float s[8], c[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    s[j] = 0.f;
    c[j] = -FLT_MAX;
    if (j < epl) {
      const int e = j * 32 + lane;
      const float lg = s_logit[warp][e];
      s[j] = 1.0f / (1.0f + expf(-lg));
      c[j] = s[j] + a.bias[e];
    }
  }

  // group score: top-1 + top-2 choice score inside each S-lane segment
  float gs_reg[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float m1 = c[j], m2 = -FLT_MAX;
    for (int o = S >> 1; o >= 1; o >>= 1) {
      const float b1 = __shfl_xor_sync(kFull, m1, o);
      const float b2 = __shfl_xor_sync(kFull, m2, o);
      const float n1 = fmaxf(m1, b1);
      const float n2 = fmaxf(fminf(m1, b1), fmaxf(m2, b2));
      m1 = n1;
      m2 = n2;
    }
    gs_reg[j] = m1 + m2;
  }
  // lane g (< G) takes group g's score
  float my_gs = -FLT_MAX;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float v = __shfl_sync(kFull, gs_reg[j], (lane * S) & 31);
    if (lane < a.G && ((lane * S) >> 5) == j) my_gs = v;
  }
  // keep the best kg groups: (score desc, group asc)
  uint32_t keep_mask = 0;
  bool kept = false;
  for (int r = 0; r < a.kg; ++r) {
    const bool cand = lane < a.G && !kept;
    float v = cand ? my_gs : -FLT_MAX;
    int id = cand ? lane : (1 << 30);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, v, o);
      const int oi = __shfl_xor_sync(kFull, id, o);
      if (ov > v || (ov == v && oi < id)) {
        v = ov;
        id = oi;
      }
    }
    if (lane == id) kept = true;
    keep_mask |= 1u << (id & 31);
  }
  // top-k experts of the kept groups: (choice score desc, expert asc)
  uint32_t taken = 0;
  int slot_e = 0;
  float slot_s = 0.f;
  for (int r = 0; r < a.k; ++r) {
    float bv = -FLT_MAX;
    int be = 1 << 30;
    float bs = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < epl) {
        const int e = j * 32 + lane;
        const bool el = ((keep_mask >> (e / S)) & 1u) && !((taken >> j) & 1u);
        if (el && (c[j] > bv || (c[j] == bv && e < be))) {
          bv = c[j];
          be = e;
          bs = s[j];
        }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oe = __shfl_xor_sync(kFull, be, o);
      const float os = __shfl_xor_sync(kFull, bs, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
        bs = os;
      }
    }
    if ((be & 31) == lane) taken |= 1u << ((be >> 5) & 31);
    if (lane == r) {
      slot_e = be;
      slot_s = bs;
    }
  }
  // renormalise over the sigmoid scores in slot order, times the routed scale
  double ssum = 0.0;
  for (int r = 0; r < a.k; ++r) ssum += static_cast<double>(__shfl_sync(kFull, slot_s, r));
  if (lane < a.k) {
    a.idx[t * a.k + lane] = slot_e;
    a.w[t * a.k + lane] =
        static_cast<float>(static_cast<double>(a.alpha) * static_cast<double>(slot_s) / ssum);
  }
}

// ------------------------------------------------------------ router split
// planes[e] = for each 64-wide K range r: [hi | mid | lo] of that range, with
// hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid): each product with
// a BF16 x is exact in FP32, and hi + mid + lo equals w to within 2^-24
// relative.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ w, int32_t E,
                                                           int32_t d, uint16_t* __restrict__ planes) {
  const int64_t n = static_cast<int64_t>(E) * d;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i / d, j = i % d;
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    uint16_t* blk = planes + e * 3 * d + (j / 64) * 192 + (j % 64);
    blk[0] = *reinterpret_cast<const uint16_t*>(&hi);
    blk[64] = *reinterpret_cast<const uint16_t*>(&mid);
    blk[128] = *reinterpret_cast<const uint16_t*>(&lo);
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

__global__ void __launch_bounds__(256) permute_kernel(PermuteArgs a) {
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  __shared__ int s_cnt[8], s_below[8], s_warp[8];
  __shared__ int s_tot[2];
  constexpr int64_t kStep = 256 * kPermPer;

  int cnt = 0, below = 0;
  for (int64_t base = 0; base < a.TK; base += kStep) {
    const int64_t i0 = base + static_cast<int64_t>(tid) * kPermPer;
    if (i0 >= a.TK) continue;
    int v[kPermPer];
    load8(a.idx, i0, a.TK, v);
#pragma unroll
    for (int j = 0; j < kPermPer; ++j) {
      if (i0 + j >= a.TK) break;
      if (static_cast<unsigned>(v[j]) >= static_cast<unsigned>(a.E)) {
        if (e == 0) {
          a.pair_row[i0 + j] = -1;
          latch_status(a.status, kStatusDeviceCheck);
        }
        continue;
      }
      cnt += (v[j] == e);
      below += (v[j] < e);
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
  int running = 0;
  for (int64_t base = 0; base < a.TK && running < total; base += kStep) {
    const int64_t i0 = base + static_cast<int64_t>(tid) * kPermPer;
    int v[kPermPer];
    if (i0 < a.TK) {
      load8(a.idx, i0, a.TK, v);
    } else {
#pragma unroll
      for (int j = 0; j < kPermPer; ++j) v[j] = -1;
    }
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
        a.perm_src[row] = static_cast<int>(i);
        a.pair_row[i] = row;
        a.perm_w[row] = a.w[i];
        ++row;
      }
    }
    running += tot;
    __syncthreads();
  }
}

// ------------------------------------------------------------------ gather
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
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = src[i];
}

// ----------------------------------------------------------------- combine
// out[t] = bf16( sum over slots, in slot order, of y[row(t, slot)] ) in FP32.
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ y,
                                                      const int32_t* __restrict__ pair_row,
                                                      int32_t k, int32_t d,
                                                      uint16_t* __restrict__ out) {
  const int64_t t = blockIdx.x;
  const int c8 = blockIdx.y * blockDim.x + threadIdx.x;
  if (c8 >= d / 8) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int sl = 0; sl < k; ++sl) {
    const int row = pair_row[t * k + sl];
    if (row < 0) continue;
    const float4* src = reinterpret_cast<const float4*>(y + static_cast<int64_t>(row) * d) + 2 * c8;
    const float4 a = src[0];
    const float4 b = src[1];
    acc[0] += a.x;
    acc[1] += a.y;
    acc[2] += a.z;
    acc[3] += a.w;
    acc[4] += b.x;
    acc[5] += b.y;
    acc[6] += b.z;
    acc[7] += b.w;
  }
  uint4 o;
  uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    ow[i] = static_cast<uint32_t>(f32_to_bf16(acc[2 * i])) |
            (static_cast<uint32_t>(f32_to_bf16(acc[2 * i + 1])) << 16);
  reinterpret_cast<uint4*>(out + t * d)[c8] = o;
}

}  // namespace

void launch_router(const RouterArgs& a, int ksplit, cudaStream_t s) {
  dim3 grid((a.E + kRtExp - 1) / kRtExp, static_cast<unsigned>((a.T + kRtTok - 1) / kRtTok), ksplit);
  router_kernel<<<grid, 256, 0, s>>>(a);
}

void launch_select(const SelectArgs& a, cudaStream_t s) {
  // one token per block while split-K partials need reducing, else 8
  const int tpb = a.ksplit > 1 ? 1 : kSelMaxTok;
  select_kernel<<<static_cast<unsigned>((a.T + tpb - 1) / tpb), 256, 0, s>>>(a, tpb);
}

void launch_router_split(const float* w, int32_t E, int32_t d, uint16_t* planes, cudaStream_t s) {
  router_split_kernel<<<512, 256, 0, s>>>(w, E, d, planes);
}

void launch_permute(const PermuteArgs& a, cudaStream_t s) {
  permute_kernel<<<a.E, 256, 0, s>>>(a);
}

void launch_gather(const uint16_t* x, const int32_t* perm_src, const int32_t* n_valid, int64_t TK,
                   int32_t k, int32_t d, uint16_t* x_perm, cudaStream_t s) {
  gather_kernel<<<static_cast<unsigned>(TK), 128, 0, s>>>(x, perm_src, n_valid, k, d, x_perm);
}

void launch_combine(const float* y, const int32_t* pair_row, int64_t T, int32_t k, int32_t d,
                    uint16_t* out, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(T), (d / 8 + 127) / 128);
  combine_kernel<<<grid, 128, 0, s>>>(y, pair_row, k, d, out);
}

}  // namespace beam
