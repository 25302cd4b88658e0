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
// x 4 experts, FP32 FMA in ascending K order (fixed order => deterministic).
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

  for (int kc = k_begin; kc < k_end; kc += kRtK) {
    {  // x tile: 32 tokens x 32 k, 4 bf16 per thread
      const int r = tid >> 3;
      const int c = (tid & 7) * 4;
      const int64_t t = t0 + r;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < a.T) {
        const uint2 raw = *reinterpret_cast<const uint2*>(a.x + t * a.d + kc + c);
        v[0] = bf16_to_f32(static_cast<uint16_t>(raw.x & 0xffffu));
        v[1] = bf16_to_f32(static_cast<uint16_t>(raw.x >> 16));
        v[2] = bf16_to_f32(static_cast<uint16_t>(raw.y & 0xffffu));
        v[3] = bf16_to_f32(static_cast<uint16_t>(raw.y >> 16));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) xs[c + i][r] = v[i];
    }
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {  // W tile: 64 experts x 32 k
      const int li = tid + rep * 256;
      const int r = li >> 3;
      const int c = (li & 7) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + r < a.E)
        v = *reinterpret_cast<const float4*>(a.w + static_cast<int64_t>(e0 + r) * a.d + kc + c);
      ws[c + 0][r] = v.x;
      ws[c + 1][r] = v.y;
      ws[c + 2][r] = v.z;
      ws[c + 3][r] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kRtK; ++kk) {
      const float x0 = xs[kk][ty * 2];
      const float x1 = xs[kk][ty * 2 + 1];
      const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      acc[0][0] = fmaf(x0, wv.x, acc[0][0]);
      acc[0][1] = fmaf(x0, wv.y, acc[0][1]);
      acc[0][2] = fmaf(x0, wv.z, acc[0][2]);
      acc[0][3] = fmaf(x0, wv.w, acc[0][3]);
      acc[1][0] = fmaf(x1, wv.x, acc[1][0]);
      acc[1][1] = fmaf(x1, wv.y, acc[1][1]);
      acc[1][2] = fmaf(x1, wv.z, acc[1][2]);
      acc[1][3] = fmaf(x1, wv.w, acc[1][3]);
    }
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
// One warp per token.  Lane l holds experts j*32 + l (j < E/32).  Groups are
// S = E/G consecutive experts, S a power of two <= 32, so a group is an
// aligned segment of S lanes of one register.
__global__ void __launch_bounds__(256) select_kernel(SelectArgs a) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (t >= a.T) return;
  const int E = a.E;
  const int epl = E >> 5;
  const int S = E / a.G;

  float s[8], c[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    s[j] = 0.f;
    c[j] = -FLT_MAX;
    if (j < epl) {
      const int e = j * 32 + lane;
      float lg = a.part[t * E + e];
      for (int sp = 1; sp < a.ksplit; ++sp) lg += a.part[(static_cast<int64_t>(sp) * a.T + t) * E + e];
      if (a.logits) a.logits[t * E + e] = lg;
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

// ----------------------------------------------------------------- permute
// Block e: counts its rows, finds its first permuted row (entries with a
// smaller expert index) and writes its rows in (token, slot) order.
__global__ void __launch_bounds__(256) permute_kernel(PermuteArgs a) {
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  __shared__ int s_cnt[8], s_below[8], s_warp[8];
  __shared__ int s_tot[2];

  int cnt = 0, below = 0;
  for (int64_t i = tid; i < a.TK; i += 256) {
    const int v = a.idx[i];
    if (static_cast<unsigned>(v) >= static_cast<unsigned>(a.E)) {
      if (e == 0) {
        a.pair_row[i] = -1;
        latch_status(a.status, kStatusDeviceCheck);
      }
      continue;
    }
    cnt += (v == e);
    below += (v < e);
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
  for (int64_t base = 0; base < a.TK && running < total; base += 256) {
    const int64_t i = base + tid;
    const bool f = (i < a.TK) && (a.idx[i] == e);
    const unsigned m = __ballot_sync(kFull, f);
    const int wpre = __popc(m & ((1u << lane) - 1u));
    if (lane == 0) s_warp[warp] = __popc(m);
    __syncthreads();
    int woff = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int cw = s_warp[w];
      woff += (w < warp) ? cw : 0;
      tot += cw;
    }
    if (f) {
      const int row = first + running + woff + wpre;
      a.perm_src[row] = static_cast<int>(i);
      a.pair_row[i] = row;
      a.perm_w[row] = a.w[i];
    }
    running += tot;
    __syncthreads();
  }
}

// ------------------------------------------------------------------ gather
// x_perm[row] = x[token of row]; rows past the last valid one are skipped.
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
  select_kernel<<<static_cast<unsigned>((a.T + 7) / 8), 256, 0, s>>>(a);
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
