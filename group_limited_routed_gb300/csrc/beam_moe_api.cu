// Host side of the C ABI declared in include/beam_moe.h: argument checks,
// workspace carve-up, tensor-map encoding and the launch sequence on the
// caller's stream.  No allocation, no host/device synchronisation (except in
// beam_moe_check_status).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/beam_moe.h"
#include "common.cuh"
#include "expert_gemm.cuh"

namespace {

using beam::GemmArgs;

constexpr size_t kAlign = 256;
constexpr int kMinRows = 256;  // token-operand buffers hold at least one full tile
constexpr int64_t kTensorRouterMinT = 256;  // from here on the router runs on tensor cores
// SM count the router's split-K partials are sized for (a workspace is sized
// without a device); a call on a larger GPU splits no further than that room
constexpr int kSizingSms = 160;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// ---------------------------------------------------------------- settings
cudaEvent_t g_events[8];
int g_num_events = 0;
uint64_t g_wait_ns = kDefaultWaitNs;
int g_withhold = 0;

// ---------------------------------------------------------------- driver entry
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

bool encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode != nullptr;
}

// 2-D BF16 tensor [rows, cols] (cols contiguous), box {64, box_rows}, 128-byte swizzle.
bool tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 2-D byte tensor [rows, cols], box {box_cols, box_rows}; 128-byte swizzle
// when box_cols is 128, none otherwise.
bool tmap_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
             uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// ---------------------------------------------------------------- device facts
struct DevInfo {
  int sms = 0;
  bool supported = false;
};

bool device_info(DevInfo* out) {
  static DevInfo cache[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev].sms == 0) {
    int sms = 0, major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return false;
    cache[dev].sms = sms;
    cache[dev].supported = (major == 10 && minor == 3);
  }
  *out = cache[dev];
  return true;
}

// ---------------------------------------------------------------- shapes
bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

bool valid_cfg(const beam_moe_config_t* c) {
  if (!c) return false;
  if (c->d <= 0 || c->d % 128 || c->d_ff <= 0 || c->d_ff % 128) return false;
  if (c->n_experts <= 0 || c->n_experts % 32 || c->n_experts > 256) return false;
  if (c->n_groups <= 0 || c->n_experts % c->n_groups) return false;
  const int S = c->n_experts / c->n_groups;
  if (S < 2 || S > 32 || !is_pow2(S)) return false;
  if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return false;
  if (c->topk < 1 || c->topk > 32 || c->topk > c->topk_groups * S) return false;
  if (!(c->routed_scale > 0.f)) return false;
  return true;
}

int router_ksplit(const beam_moe_config_t& c, int64_t T) {
  const int64_t blocks = static_cast<int64_t>((c.n_experts + 63) / 64) * ((T + 31) / 32);
  const int64_t want = (2 * 152 + blocks - 1) / std::max<int64_t>(blocks, 1);
  const int64_t ks = std::max<int64_t>(1, std::min<int64_t>(c.d / 128, want));
  // K range per split, a multiple of 32
  const int64_t chunk = ((c.d + ks - 1) / ks + 31) / 32 * 32;
  return static_cast<int>((c.d + chunk - 1) / chunk);
}

int router_chunk(const beam_moe_config_t& c, int ks) {
  return static_cast<int>(((c.d + ks - 1) / ks + 31) / 32 * 32);
}

// Token-block widths of the two expert GEMMs: 16 when experts see a few rows
// each (weight streaming), else 256 for the compute-bound regime (fewer
// re-reads of each weight tile from L2).
bool small_batch(const beam_moe_config_t& c, int64_t TK) { return TK <= 4LL * c.n_experts; }
int gateup_tile(const beam_moe_config_t& c, int64_t TK) { return small_batch(c, TK) ? 16 : 256; }
int down_tile(const beam_moe_config_t& c, int64_t TK) { return small_batch(c, TK) ? 16 : 256; }

// 256-token blocks run on clusters of two CTAs sharing M = 256 MMAs
// (expert_gemm_pair_kernel.cuh) when the weight rows divide into the pair
// tiles: 256 rows of d_ff for gate/up, 512 rows of d for down.
bool pair_gateup(const beam_moe_config_t& c, int64_t TK) {
  return !small_batch(c, TK) && c.d_ff % 256 == 0;
}
bool pair_down(const beam_moe_config_t& c, int64_t TK) {
  return !small_batch(c, TK) && c.d % 512 == 0;
}

bool tensor_router(const beam_moe_config_t& c, int64_t T) {
  return T >= kTensorRouterMinT && c.n_experts % 128 == 0;
}

// Below the tensor-router threshold the router, the selection and the
// permutation run as one cooperative launch (decode-sized batches, where
// each of the three would be a few microseconds of mostly launch latency).
bool fused_routing(const beam_moe_config_t& c, int64_t T) {
  return T < kTensorRouterMinT && c.n_experts <= 256;
}

struct Layout {
  size_t status, part, logits, idx, w, counts, offsets, perm_src, pair_row, perm_w, x_perm, h, y,
      router_planes, x_fp4, x_sf, h_fp4, h_sf, x_fp8, x_scale, h_fp8, h_scale, total;
};

bool known_fmt(int32_t fmt) {
  return fmt == BEAM_WEIGHTS_BF16 || fmt == BEAM_WEIGHTS_NVFP4 || fmt == BEAM_WEIGHTS_NVFP4_A16 ||
         fmt == BEAM_WEIGHTS_FP8 || fmt == BEAM_WEIGHTS_MXFP8;
}

// NVFP4 token-block width: the token scales are read row-major, 32 rows at most
int fp4_tile(const beam_moe_config_t& c, int64_t TK) { return small_batch(c, TK) ? 16 : 32; }

Layout make_layout(const beam_moe_config_t& c, int64_t T_max, int32_t fmt = BEAM_WEIGHTS_BF16) {
  const bool fp4 = fmt == BEAM_WEIGHTS_NVFP4;
  const bool a16 = fmt == BEAM_WEIGHTS_NVFP4_A16;  // F16 token rows gathered into x_perm
  const bool fp8 = fmt == BEAM_WEIGHTS_FP8;         // E4M3 token rows (gathered when large)
  const bool mx = fmt == BEAM_WEIGHTS_MXFP8;        // MX token rows and h (codes + scales)
  const int64_t E = c.n_experts, k = c.topk;
  const int64_t TK = T_max * k;
  const int64_t rows = std::max<int64_t>(TK, kMinRows);
  int64_t part_rows = 0;  // max over T <= T_max of ksplit(T) * T
  for (int64_t nb = 1; nb <= (T_max + 31) / 32; ++nb) {
    const int64_t Tn = std::min<int64_t>(T_max, nb * 32);
    const int64_t ks = tensor_router(c, Tn)
                           ? beam::router_tc_ksplit(Tn, c.n_experts, c.d, kSizingSms)
                           : router_ksplit(c, Tn);
    part_rows = std::max<int64_t>(part_rows, ks * Tn);
  }
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  L.status = take(kAlign);
  L.part = take(static_cast<size_t>(part_rows) * E * 4);
  L.logits = take(static_cast<size_t>(T_max) * E * 4);
  L.idx = take(static_cast<size_t>(TK) * 4);
  L.w = take(static_cast<size_t>(TK) * 4);
  L.counts = take(static_cast<size_t>(E) * 4);
  L.offsets = take(static_cast<size_t>(E + 1) * 4);
  L.perm_src = take(static_cast<size_t>(TK) * 4);
  L.pair_row = take(static_cast<size_t>(TK) * 4);
  L.perm_w = take(static_cast<size_t>(TK) * 4);
  // gathered token rows: F16 (W4A16), E4M3 (FP8) or BF16, the last two only
  // for batches that do not gather inside the gate/up GEMM
  const size_t xrow = static_cast<size_t>(rows) * c.d;
  L.x_perm = take(a16 ? xrow * 2 : fp4 || mx || small_batch(c, TK) ? 0 : fp8 ? xrow : xrow * 2);
  L.h = take(fp4 || mx ? 0 : static_cast<size_t>(rows) * c.d_ff * 2);
  L.y = take(static_cast<size_t>(rows) * c.d * 4);
  L.router_planes = take(T_max >= kTensorRouterMinT ? static_cast<size_t>(E) * 3 * c.d * 2 : 0);
  // block-scaled token rows and h: NVFP4 codes (half a byte) and a scale slot
  // per 64 elements, or MXFP8 codes (a byte) and a scale slot per 128
  L.x_fp4 = take(fp4 ? static_cast<size_t>(rows) * c.d / 2 : mx ? xrow : 0);
  L.x_sf = take(fp4 ? static_cast<size_t>(rows) * c.d / 4 : mx ? xrow / 8 : 0);
  L.h_fp4 = take(fp4 ? static_cast<size_t>(rows) * c.d_ff / 2
                     : mx ? static_cast<size_t>(rows) * c.d_ff : 0);
  L.h_sf = take(fp4 ? static_cast<size_t>(rows) * c.d_ff / 4
                    : mx ? static_cast<size_t>(rows) * c.d_ff / 8 : 0);
  L.x_fp8 = take(fp8 ? static_cast<size_t>(T_max) * c.d : 0);
  L.x_scale = take(fp8 ? static_cast<size_t>(T_max) * 4 : 0);
  L.h_fp8 = take(fp8 ? static_cast<size_t>(rows) * c.d_ff : 0);
  L.h_scale = take(fp8 ? static_cast<size_t>(rows) * 4 : 0);
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// Inside a stream capture a plain record only orders streams; the external
// flag makes it an event-record node that timestamps every graph replay.
void record(int i, cudaStream_t s) {
  if (g_num_events < 8) return;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cap);
  if (cap == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(g_events[i], s, cudaEventRecordExternal);
  else
    cudaEventRecord(g_events[i], s);
}

beam_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? BEAM_OK : BEAM_ERR_CUDA; }

// BEAM_OK with *empty set for a valid call of zero tokens (nothing to check
// further, nothing to launch).
beam_status_t common_checks(const beam_moe_config_t* cfg, int64_t T, void* ws, size_t ws_bytes,
                            Layout* L, DevInfo* dev, bool* empty,
                            int32_t fmt = BEAM_WEIGHTS_BF16) {
  if (!valid_cfg(cfg) || T < 0 || T > (int64_t(1) << 31) / 64) return BEAM_ERR_INVALID_ARG;
  if ((fmt == BEAM_WEIGHTS_NVFP4 || fmt == BEAM_WEIGHTS_NVFP4_A16) && (cfg->d % 256 || cfg->d_ff % 256))
    return BEAM_ERR_INVALID_ARG;
  // the MXFP8 down GEMM takes its weight rows in pairs of 128-row blocks
  if (fmt == BEAM_WEIGHTS_MXFP8 && cfg->d % 256) return BEAM_ERR_INVALID_ARG;
  *empty = (T == 0);
  if (*empty) return BEAM_OK;
  if (!aligned16(ws)) return BEAM_ERR_INVALID_ARG;
  *L = make_layout(*cfg, T, fmt);
  if (ws_bytes < L->total) return BEAM_ERR_WORKSPACE;
  if (!device_info(dev)) return BEAM_ERR_CUDA;
  if (!dev->supported) return BEAM_ERR_UNSUPPORTED;
  return BEAM_OK;
}

beam::PermuteArgs permute_args(const beam_moe_config_t& c, const int32_t* idx, const float* w,
                               int64_t T, void* ws, const Layout& L) {
  beam::PermuteArgs pa;
  pa.idx = idx;
  pa.w = w;
  pa.TK = T * c.topk;
  pa.E = c.n_experts;
  pa.counts = at<int32_t>(ws, L.counts);
  pa.offsets = at<int32_t>(ws, L.offsets);
  pa.perm_src = at<int32_t>(ws, L.perm_src);
  pa.pair_row = at<int32_t>(ws, L.pair_row);
  pa.perm_w = at<float>(ws, L.perm_w);
  pa.status = at<uint32_t>(ws, L.status);
  pa.id_base = 0;
  return pa;
}

// From this many (token, slot) entries on, the permutation runs as a counting
// sort (one cooperative launch) instead of one block per expert scanning all
// entries; its chunk counts live in the router's partials buffer, which is
// dead once the selection has run (it holds at least T * E floats).
constexpr int64_t kSortMinEntries = 8192;

beam_status_t launch_permutation(const beam::PermuteArgs& pa, void* ws, const Layout& L,
                                 const DevInfo& dev, cudaStream_t s) {
  if (pa.TK >= kSortMinEntries && pa.E <= 256) {
    return beam::launch_permute_sort(pa, at<int32_t>(ws, L.part), dev.sms, s) == cudaSuccess
               ? BEAM_OK
               : BEAM_ERR_CUDA;
  }
  beam::launch_permute(pa, s);
  return BEAM_OK;
}

// router + selection into idx/w (and logits).  With `permuted` given and a
// decode-sized batch, the permutation runs in the same cooperative launch and
// *permuted is set.
beam_status_t run_route(const beam_moe_config_t& c, const void* hidden, const float* router_w,
                        const float* bias, int64_t T, int32_t* idx, float* w, float* logits,
                        void* ws, const Layout& L, const DevInfo& dev, cudaStream_t s,
                        bool* permuted = nullptr) {
  int ks = 1;
  float* part = at<float>(ws, L.part);
  if (permuted) *permuted = false;
  beam::RouterArgs ra;
  if (tensor_router(c, T)) {
    // BF16x3 on the tensor cores: W_r split into three BF16 planes
    uint16_t* planes = at<uint16_t>(ws, L.router_planes);
    beam::launch_router_split(router_w, c.n_experts, c.d, planes, s);
    CUtensorMap tm_w, tm_x;
    if (!tmap_bf16(&tm_w, planes, c.n_experts, 3LL * c.d, 128) ||
        !tmap_bf16(&tm_x, hidden, T, c.d, 128))
      return BEAM_ERR_CUDA;
    // splits the workspace's partials buffer has room for
    const int64_t room = static_cast<int64_t>((L.logits - L.part) / (4 * c.n_experts)) / T;
    ks = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(beam::router_tc_ksplit(T, c.n_experts, c.d, dev.sms), room)));
    if (beam::launch_router_tc(tm_w, tm_x, part, T, c.n_experts, c.d, ks,
                               at<uint32_t>(ws, L.status), g_wait_ns, dev.sms, s) != cudaSuccess)
      return BEAM_ERR_CUDA;
  } else {
    ks = router_ksplit(c, T);
    ra.x = static_cast<const uint16_t*>(hidden);
    ra.w = router_w;
    ra.part = part;
    ra.T = T;
    ra.d = c.d;
    ra.E = c.n_experts;
    ra.k_chunk = router_chunk(c, ks);
  }
  beam::SelectArgs sa;
  sa.part = part;
  sa.ksplit = ks;
  sa.bias = bias;
  sa.T = T;
  sa.E = c.n_experts;
  sa.G = c.n_groups;
  sa.kg = c.topk_groups;
  sa.k = c.topk;
  sa.alpha = c.routed_scale;
  sa.idx = idx;
  sa.w = w;
  sa.logits = logits;
  if (!tensor_router(c, T) && permuted && fused_routing(c, T)) {
    const beam::PermuteArgs pa = permute_args(c, idx, w, T, ws, L);
    if (beam::launch_fused_route(ra, ks, sa, pa, dev.sms, s) != cudaSuccess) return BEAM_ERR_CUDA;
    *permuted = true;
    record(1, s);
    record(2, s);
    record(3, s);
    return BEAM_OK;
  }
  if (!tensor_router(c, T)) beam::launch_router(ra, ks, s);
  record(1, s);
  beam::launch_select(sa, s);
  record(2, s);
  return cuda_status(cudaGetLastError());
}

// The layer's last kernel: the weighted combine of the FP32 expert rows y
// into BF16 out, or that combine followed by the sublayer boundary when one
// is given (every expert format ends in the same y rows).  With y_pairs
// given (expert parallelism) there is no combine here.
cudaError_t finish_combine(const beam_moe_config_t& c, const float* y, const int32_t* pair_row,
                           int64_t T, void* out, const float* y_pairs,
                           const beam::BoundaryArgs* boundary, uint32_t* status, cudaStream_t s) {
  if (y_pairs) return cudaSuccess;
  if (boundary)
    return beam::launch_combine_boundary(y, pair_row, T, c.topk, c.d,
                                         static_cast<uint16_t*>(out), *boundary, status, s);
  beam::launch_combine(y, pair_row, T, c.topk, c.d, static_cast<uint16_t*>(out), status, s);
  return cudaGetLastError();
}

// permute + gather + expert GEMMs + combine.  With y_pairs given, the down
// GEMM writes each pair's weighted FP32 row there (pair order) and there is
// no combine; idx then holds ids from id_base on.
beam_status_t run_experts(const beam_moe_config_t& c, const void* hidden, const int32_t* idx,
                          const float* w, const void* w_gate, const void* w_up,
                          const void* w_down, void* out, int64_t T, void* ws, const Layout& L,
                          const DevInfo& dev, cudaStream_t s, bool permuted = false,
                          float* y_pairs = nullptr, int32_t id_base = 0,
                          const beam::BoundaryArgs* boundary = nullptr) {
  const int64_t TK = T * c.topk;
  const int64_t rows = std::max<int64_t>(TK, kMinRows);
  const int nt_gu = gateup_tile(c, TK);
  const int nt_dn = down_tile(c, TK);
  uint32_t* status = at<uint32_t>(ws, L.status);

  beam::PermuteArgs pa = permute_args(c, idx, w, T, ws, L);
  pa.id_base = id_base;
  if (!permuted) {
    if (launch_permutation(pa, ws, L, dev, s) != BEAM_OK) return BEAM_ERR_CUDA;
    record(3, s);
  }
  // decode-sized batches: the gate/up GEMM gathers its token rows itself
  const bool row_gather = small_batch(c, TK);
  uint16_t* xp = at<uint16_t>(ws, L.x_perm);
  if (!row_gather)
    beam::launch_scatter_tokens(static_cast<const uint16_t*>(hidden), pa.pair_row, T, c.topk, c.d,
                                xp, status, s);
  record(4, s);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return BEAM_ERR_CUDA;

  const int64_t EF = static_cast<int64_t>(c.n_experts) * c.d_ff;
  const int64_t ED = static_cast<int64_t>(c.n_experts) * c.d;
  uint16_t* h = at<uint16_t>(ws, L.h);
  float* y = at<float>(ws, L.y);
  CUtensorMap tm_wg, tm_wu, tm_wd, tm_xp, tm_h;
  // token boxes: one row (row gather), a whole block, or half a block for
  // the CTA pairs
  const bool pgu = pair_gateup(c, TK), pdn = pair_down(c, TK);
  if (!tmap_bf16(&tm_wg, w_gate, EF, c.d, 128) || !tmap_bf16(&tm_wu, w_up, EF, c.d, 128) ||
      !tmap_bf16(&tm_wd, w_down, ED, c.d_ff, 128) || !(row_gather ? tmap_bf16(&tm_xp, hidden, T, c.d, 1)
                  : tmap_bf16(&tm_xp, xp, rows, c.d, pgu ? nt_gu / 2 : nt_gu)) ||
      !tmap_bf16(&tm_h, h, rows, c.d_ff, pdn ? nt_dn / 2 : nt_dn))
    return BEAM_ERR_CUDA;

  GemmArgs ga{};
  ga.counts = pa.counts;
  ga.perm_src = pa.perm_src;
  ga.topk = c.topk;
  ga.offsets = pa.offsets;
  ga.perm_w = pa.perm_w;
  ga.E = c.n_experts;
  ga.status = status;
  ga.wait_limit_ns = g_wait_ns;
  ga.withhold_first_load = g_withhold;
  ga.weight_evict_first = small_batch(c, TK) ? 1 : 0;
  g_withhold = 0;

  // upper bound of the tile count, to size the persistent grid
  auto grid_for = [&](int m_blocks, int nt) {
    const int64_t tiles = static_cast<int64_t>(m_blocks) * (c.n_experts + (TK + nt - 1) / nt);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev.sms, tiles)));
  };

  ga.h_out = h;
  ga.out_ld = c.d_ff;
  ga.rows_per_expert = c.d_ff;
  ga.m_blocks = c.d_ff / 128;
  ga.k_blocks = c.d / 64;
  ga.b_k_blocks = ga.k_blocks;
  ga.a_rows = static_cast<int32_t>(EF);
  ga.b_rows = static_cast<int32_t>(row_gather ? T : rows);
  ga.out_rows_cap = static_cast<int32_t>(rows);
  if (pgu) {
    ga.m_blocks = c.d_ff / 256;
    err = beam::launch_grouped_gemm_pair(true, tm_wg, tm_wu, tm_xp, ga,
                                         grid_for(ga.m_blocks, nt_gu), s);
  } else {
    err = beam::launch_grouped_gemm(beam::kModeGateUp, nt_gu, tm_wg, tm_wu, tm_xp, ga,
                                    grid_for(ga.m_blocks, nt_gu), s);
  }
  if (err != cudaSuccess) return BEAM_ERR_CUDA;
  record(5, s);

  ga.withhold_first_load = 0;
  ga.h_out = nullptr;
  ga.f32_out = y_pairs ? y_pairs : y;
  ga.out_rows = y_pairs ? pa.perm_src : nullptr;
  ga.out_ld = c.d;
  ga.rows_per_expert = c.d;
  // 256-token blocks: pairs of adjacent 128-row W_d blocks share one token
  // tile (half the token-tile reads per flop); decode-sized blocks stay single
  const bool pair = c.d % 256 == 0 && nt_dn == 256;
  ga.m_blocks = pair ? c.d / 256 : c.d / 128;
  ga.k_blocks = c.d_ff / 64;
  ga.b_k_blocks = ga.k_blocks;
  ga.a_rows = static_cast<int32_t>(ED);
  ga.b_rows = static_cast<int32_t>(rows);
  ga.out_rows_cap = static_cast<int32_t>(y_pairs ? TK : rows);
  if (pdn) {
    ga.m_blocks = c.d / 512;
    err = beam::launch_grouped_gemm_pair(false, tm_wd, tm_wd, tm_h, ga,
                                         grid_for(ga.m_blocks, nt_dn), s);
  } else {
    err = beam::launch_grouped_gemm(pair ? beam::kModeDownPair : beam::kModeDown, nt_dn, tm_wd,
                                    tm_wd, tm_h, ga, grid_for(ga.m_blocks, nt_dn), s);
  }
  if (err != cudaSuccess) return BEAM_ERR_CUDA;
  record(6, s);

  if (finish_combine(c, y, pa.pair_row, T, out, y_pairs, boundary, pa.status, s) != cudaSuccess)
    return BEAM_ERR_CUDA;
  record(7, s);
  return cuda_status(cudaGetLastError());
}

// permute + quantise token rows + FP4 gate/up (quantising h) + FP4 down + combine
// With y_pairs given, the down GEMM writes each pair's weighted FP32 row there
// (pair order) and there is no combine; idx then holds ids from id_base on.
beam_status_t run_experts_nvfp4(const beam_moe_config_t& c, const void* hidden, const int32_t* idx,
                                const float* w, const beam_fp4_weight_t& gate,
                                const beam_fp4_weight_t& up, const beam_fp4_weight_t& down,
                                void* out, int64_t T, void* ws, const Layout& L,
                                const DevInfo& dev, cudaStream_t s, bool permuted = false,
                                float* y_pairs = nullptr, int32_t id_base = 0,
                                const beam::BoundaryArgs* boundary = nullptr) {
  const int64_t TK = T * c.topk;
  const int64_t rows = std::max<int64_t>(TK, kMinRows);
  const int nt = fp4_tile(c, TK);
  uint32_t* status = at<uint32_t>(ws, L.status);
  beam::PermuteArgs pa = permute_args(c, idx, w, T, ws, L);
  pa.id_base = id_base;
  if (!permuted) {
    if (launch_permutation(pa, ws, L, dev, s) != BEAM_OK) return BEAM_ERR_CUDA;
    record(3, s);
  }
  uint8_t* xq = at<uint8_t>(ws, L.x_fp4);
  uint8_t* xsf = at<uint8_t>(ws, L.x_sf);
  uint8_t* hq = at<uint8_t>(ws, L.h_fp4);
  uint8_t* hsf = at<uint8_t>(ws, L.h_sf);
  float* y = at<float>(ws, L.y);
  beam::launch_quantize_tokens(static_cast<const uint16_t*>(hidden), pa.pair_row, T, c.topk, c.d,
                               xq, xsf, status, s);
  record(4, s);
  if (cudaGetLastError() != cudaSuccess) return BEAM_ERR_CUDA;

  const int64_t EF = static_cast<int64_t>(c.n_experts) * c.d_ff;
  const int64_t ED = static_cast<int64_t>(c.n_experts) * c.d;
  CUtensorMap tm_g, tm_u, tm_d, tm_x, tm_xsf, tm_h, tm_hsf;
  if (!tmap_u8(&tm_g, gate.q, EF, c.d / 2, 128, 128) ||
      !tmap_u8(&tm_u, up.q, EF, c.d / 2, 128, 128) ||
      !tmap_u8(&tm_d, down.q, ED, c.d_ff / 2, 128, 128) ||
      !tmap_u8(&tm_x, xq, rows, c.d / 2, 128, nt) || !tmap_u8(&tm_xsf, xsf, rows, c.d / 4, 16, 32) ||
      !tmap_u8(&tm_h, hq, rows, c.d_ff / 2, 128, nt) ||
      !tmap_u8(&tm_hsf, hsf, rows, c.d_ff / 4, 16, 32))
    return BEAM_ERR_CUDA;
  beam::Fp4GemmArgs fa{};
  fa.counts = pa.counts;
  fa.offsets = pa.offsets;
  fa.perm_w = pa.perm_w;
  fa.E = c.n_experts;
  fa.status = status;
  fa.wait_limit_ns = g_wait_ns;
  fa.weight_evict_first = small_batch(c, TK) ? 1 : 0;
  auto grid_for = [&](int m_blocks) {
    const int64_t tiles = static_cast<int64_t>(m_blocks) * (c.n_experts + (TK + nt - 1) / nt);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev.sms, tiles)));
  };
  fa.sfa0 = gate.sf;
  fa.sfa1 = up.sf;
  fa.gs0 = gate.global_scale;
  fa.gs1 = up.global_scale;
  fa.hq = hq;
  fa.hsf = hsf;
  fa.out_ld = c.d_ff;
  fa.rows_per_expert = c.d_ff;
  fa.m_blocks = c.d_ff / 128;
  fa.k_blocks = c.d / 256;
  fa.a_rows = static_cast<int32_t>(EF);
  fa.b_rows = static_cast<int32_t>(rows);
  fa.out_rows_cap = static_cast<int32_t>(rows);
  if (beam::launch_fp4_gemm(true, nt, tm_g, tm_u, tm_x, tm_xsf, fa, grid_for(fa.m_blocks), s) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  record(5, s);
  fa.sfa0 = down.sf;
  fa.sfa1 = nullptr;
  fa.gs0 = down.global_scale;
  fa.gs1 = nullptr;
  fa.hq = nullptr;
  fa.hsf = nullptr;
  fa.y = y_pairs ? y_pairs : y;
  fa.out_rows = y_pairs ? pa.perm_src : nullptr;
  fa.out_ld = c.d;
  fa.rows_per_expert = c.d;
  fa.m_blocks = c.d / 256;  // pairs of 128-row weight blocks
  fa.k_blocks = c.d_ff / 256;
  fa.a_rows = static_cast<int32_t>(ED);
  fa.out_rows_cap = static_cast<int32_t>(y_pairs ? TK : rows);
  if (beam::launch_fp4_gemm(false, nt, tm_d, tm_d, tm_h, tm_hsf, fa, grid_for(fa.m_blocks), s) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  record(6, s);
  if (finish_combine(c, y, pa.pair_row, T, out, y_pairs, boundary, pa.status, s) != cudaSuccess)
    return BEAM_ERR_CUDA;
  record(7, s);
  return cuda_status(cudaGetLastError());
}

// permute + MX token rows + MXFP8 gate/up (quantising h to MX) + MXFP8 down
// + combine
beam_status_t run_experts_mxfp8(const beam_moe_config_t& c, const void* hidden, const int32_t* idx,
                                const float* w, const beam_mxfp8_weight_t& gate,
                                const beam_mxfp8_weight_t& up, const beam_mxfp8_weight_t& down,
                                void* out, int64_t T, void* ws, const Layout& L,
                                const DevInfo& dev, cudaStream_t s, bool permuted = false,
                                const beam::BoundaryArgs* boundary = nullptr) {
  const int64_t TK = T * c.topk;
  const int64_t rows = std::max<int64_t>(TK, kMinRows);
  const int nt = fp4_tile(c, TK);
  const beam::PermuteArgs pa = permute_args(c, idx, w, T, ws, L);
  if (!permuted) {
    if (launch_permutation(pa, ws, L, dev, s) != BEAM_OK) return BEAM_ERR_CUDA;
    record(3, s);
  }
  uint8_t* xq = at<uint8_t>(ws, L.x_fp4);
  uint8_t* xsf = at<uint8_t>(ws, L.x_sf);
  uint8_t* hq = at<uint8_t>(ws, L.h_fp4);
  uint8_t* hsf = at<uint8_t>(ws, L.h_sf);
  float* y = at<float>(ws, L.y);
  beam::launch_quantize_tokens_mx(static_cast<const uint16_t*>(hidden), pa.pair_row, T, c.topk,
                                  c.d, xq, xsf, pa.status, s);
  record(4, s);
  if (cudaGetLastError() != cudaSuccess) return BEAM_ERR_CUDA;

  const int64_t EF = static_cast<int64_t>(c.n_experts) * c.d_ff;
  const int64_t ED = static_cast<int64_t>(c.n_experts) * c.d;
  CUtensorMap tm_g, tm_u, tm_d, tm_x, tm_xsf, tm_h, tm_hsf;
  if (!tmap_u8(&tm_g, gate.q, EF, c.d, 128, 128) || !tmap_u8(&tm_u, up.q, EF, c.d, 128, 128) ||
      !tmap_u8(&tm_d, down.q, ED, c.d_ff, 128, 128) || !tmap_u8(&tm_x, xq, rows, c.d, 128, nt) ||
      !tmap_u8(&tm_xsf, xsf, rows, c.d / 8, 16, 32) ||
      !tmap_u8(&tm_h, hq, rows, c.d_ff, 128, nt) ||
      !tmap_u8(&tm_hsf, hsf, rows, c.d_ff / 8, 16, 32))
    return BEAM_ERR_CUDA;
  beam::Fp4GemmArgs fa{};
  fa.counts = pa.counts;
  fa.offsets = pa.offsets;
  fa.perm_w = pa.perm_w;
  fa.E = c.n_experts;
  fa.status = at<uint32_t>(ws, L.status);
  fa.wait_limit_ns = g_wait_ns;
  fa.weight_evict_first = small_batch(c, TK) ? 1 : 0;
  auto grid_for = [&](int m_blocks) {
    const int64_t tiles = static_cast<int64_t>(m_blocks) * (c.n_experts + (TK + nt - 1) / nt);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev.sms, tiles)));
  };
  fa.sfa0 = gate.sf;
  fa.sfa1 = up.sf;
  fa.hq = hq;
  fa.hsf = hsf;
  fa.out_ld = c.d_ff;
  fa.rows_per_expert = c.d_ff;
  fa.m_blocks = c.d_ff / 128;
  fa.k_blocks = c.d / 128;
  fa.a_rows = static_cast<int32_t>(EF);
  fa.b_rows = static_cast<int32_t>(rows);
  fa.out_rows_cap = static_cast<int32_t>(rows);
  if (beam::launch_mxfp8_gemm(true, nt, tm_g, tm_u, tm_x, tm_xsf, fa, grid_for(fa.m_blocks), s) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  record(5, s);
  fa.sfa0 = down.sf;
  fa.sfa1 = nullptr;
  fa.hq = nullptr;
  fa.hsf = nullptr;
  fa.y = y;
  fa.out_ld = c.d;
  fa.rows_per_expert = c.d;
  fa.m_blocks = c.d / 256;  // pairs of 128-row weight blocks
  fa.k_blocks = c.d_ff / 128;
  fa.a_rows = static_cast<int32_t>(ED);
  fa.out_rows_cap = static_cast<int32_t>(rows);
  if (beam::launch_mxfp8_gemm(false, nt, tm_d, tm_d, tm_h, tm_hsf, fa, grid_for(fa.m_blocks), s) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  record(6, s);
  if (finish_combine(c, y, pa.pair_row, T, out, nullptr, boundary, pa.status, s) != cudaSuccess)
    return BEAM_ERR_CUDA;
  record(7, s);
  return cuda_status(cudaGetLastError());
}

// permute + E4M3 token rows (+ gather) + FP8 gate/up (BF16 h) + E4M3 h rows
// + FP8 down + combine.  With y_pairs given, the down GEMM writes each
// pair's weighted FP32 row there (pair order) and there is no combine; idx
// then holds ids from id_base on.
beam_status_t run_experts_fp8(const beam_moe_config_t& c, const void* hidden, const int32_t* idx,
                              const float* w, const beam_fp8_weight_t& gate,
                              const beam_fp8_weight_t& up, const beam_fp8_weight_t& down,
                              void* out, int64_t T, void* ws, const Layout& L, const DevInfo& dev,
                              cudaStream_t s, bool permuted = false, float* y_pairs = nullptr,
                              int32_t id_base = 0, const beam::BoundaryArgs* boundary = nullptr) {
  const int64_t TK = T * c.topk;
  const int64_t rows = std::max<int64_t>(TK, kMinRows);
  const int nt_gu = gateup_tile(c, TK);
  const int nt_dn = down_tile(c, TK);
  beam::PermuteArgs pa = permute_args(c, idx, w, T, ws, L);
  pa.id_base = id_base;
  if (!permuted) {
    if (launch_permutation(pa, ws, L, dev, s) != BEAM_OK) return BEAM_ERR_CUDA;
    record(3, s);
  }
  // the token rows are quantised once per token; decode-sized batches gather
  // them inside the gate/up GEMM, larger ones are scattered into expert order
  // first (byte rows, copied as d/2 16-bit words)
  uint8_t* xq = at<uint8_t>(ws, L.x_fp8);
  float* xs = at<float>(ws, L.x_scale);
  beam::launch_quantize_e4m3_rows(static_cast<const uint16_t*>(hidden), nullptr, T, c.d, xq, xs,
                                  s);
  const bool row_gather = small_batch(c, TK);
  uint8_t* xp = at<uint8_t>(ws, L.x_perm);
  if (!row_gather)
    beam::launch_scatter_tokens(reinterpret_cast<const uint16_t*>(xq), pa.pair_row, T, c.topk,
                                c.d / 2, reinterpret_cast<uint16_t*>(xp), pa.status, s);
  record(4, s);
  if (cudaGetLastError() != cudaSuccess) return BEAM_ERR_CUDA;

  const int64_t EF = static_cast<int64_t>(c.n_experts) * c.d_ff;
  const int64_t ED = static_cast<int64_t>(c.n_experts) * c.d;
  uint16_t* h = at<uint16_t>(ws, L.h);
  uint8_t* hq = at<uint8_t>(ws, L.h_fp8);
  float* hs = at<float>(ws, L.h_scale);
  float* y = at<float>(ws, L.y);
  CUtensorMap tm_g, tm_u, tm_d, tm_x, tm_h;
  const bool pgu = pair_gateup(c, TK), pdn = pair_down(c, TK);
  if (!tmap_u8(&tm_g, gate.q, EF, c.d, 128, 128) || !tmap_u8(&tm_u, up.q, EF, c.d, 128, 128) ||
      !tmap_u8(&tm_d, down.q, ED, c.d_ff, 128, 128) ||
      !(row_gather ? tmap_u8(&tm_x, xq, T, c.d, 128, 1)
                   : tmap_u8(&tm_x, xp, rows, c.d, 128, pgu ? nt_gu / 2 : nt_gu)) ||
      !tmap_u8(&tm_h, hq, rows, c.d_ff, 128, pdn ? nt_dn / 2 : nt_dn))
    return BEAM_ERR_CUDA;

  GemmArgs ga{};
  ga.counts = pa.counts;
  ga.perm_src = pa.perm_src;
  ga.topk = c.topk;
  ga.offsets = pa.offsets;
  ga.perm_w = pa.perm_w;
  ga.E = c.n_experts;
  ga.status = at<uint32_t>(ws, L.status);
  ga.wait_limit_ns = g_wait_ns;
  ga.withhold_first_load = 0;
  ga.weight_evict_first = small_batch(c, TK) ? 1 : 0;
  auto grid_for = [&](int m_blocks, int nt) {
    const int64_t tiles = static_cast<int64_t>(m_blocks) * (c.n_experts + (TK + nt - 1) / nt);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev.sms, tiles)));
  };

  ga.h_out = h;
  ga.out_ld = c.d_ff;
  ga.rows_per_expert = c.d_ff;
  ga.m_blocks = c.d_ff / 128;
  ga.k_blocks = c.d / 128;
  ga.b_k_blocks = ga.k_blocks;
  ga.a_rows = static_cast<int32_t>(EF);
  ga.b_rows = static_cast<int32_t>(row_gather ? T : rows);
  ga.out_rows_cap = static_cast<int32_t>(rows);
  ga.a0_scale = gate.scale;
  ga.a1_scale = up.scale;
  ga.b_scale = xs;  // per token
  if (pgu) ga.m_blocks = c.d_ff / 256;
  if ((pgu ? beam::launch_grouped_gemm_pair(true, tm_g, tm_u, tm_x, ga,
                                            grid_for(ga.m_blocks, nt_gu), s, true)
           : beam::launch_grouped_gemm(beam::kModeGateUp, nt_gu, tm_g, tm_u, tm_x, ga,
                                       grid_for(ga.m_blocks, nt_gu), s, true)) != cudaSuccess)
    return BEAM_ERR_CUDA;
  record(5, s);

  beam::launch_quantize_e4m3_rows(h, pa.offsets + c.n_experts, TK, c.d_ff, hq, hs, s);
  ga.h_out = nullptr;
  ga.f32_out = y_pairs ? y_pairs : y;
  ga.out_rows = y_pairs ? pa.perm_src : nullptr;
  ga.out_ld = c.d;
  ga.rows_per_expert = c.d;
  const bool pair = c.d % 256 == 0 && nt_dn == 256;
  ga.m_blocks = pair ? c.d / 256 : c.d / 128;
  ga.k_blocks = c.d_ff / 128;
  ga.b_k_blocks = ga.k_blocks;
  ga.a_rows = static_cast<int32_t>(ED);
  ga.b_rows = static_cast<int32_t>(rows);
  ga.out_rows_cap = static_cast<int32_t>(y_pairs ? TK : rows);
  ga.a0_scale = down.scale;
  ga.a1_scale = nullptr;
  ga.b_scale = hs;  // per permuted row
  if (pdn) ga.m_blocks = c.d / 512;
  if ((pdn ? beam::launch_grouped_gemm_pair(false, tm_d, tm_d, tm_h, ga,
                                            grid_for(ga.m_blocks, nt_dn), s, true)
           : beam::launch_grouped_gemm(pair ? beam::kModeDownPair : beam::kModeDown, nt_dn, tm_d,
                                       tm_d, tm_h, ga, grid_for(ga.m_blocks, nt_dn), s, true)) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  record(6, s);
  if (finish_combine(c, y, pa.pair_row, T, out, y_pairs, boundary, pa.status, s) != cudaSuccess)
    return BEAM_ERR_CUDA;
  record(7, s);
  return cuda_status(cudaGetLastError());
}

// permute + F16 token rows + W4A16 gate/up (F16 h) + W4A16 down + combine
beam_status_t run_experts_w4a16(const beam_moe_config_t& c, const void* hidden, const int32_t* idx,
                                const float* w, const beam_fp4_weight_t& gate,
                                const beam_fp4_weight_t& up, const beam_fp4_weight_t& down,
                                void* out, int64_t T, void* ws, const Layout& L,
                                const DevInfo& dev, cudaStream_t s, bool permuted = false,
                                const beam::BoundaryArgs* boundary = nullptr) {
  const int64_t TK = T * c.topk;
  const int64_t rows = std::max<int64_t>(TK, kMinRows);
  const int nt = fp4_tile(c, TK);
  const beam::PermuteArgs pa = permute_args(c, idx, w, T, ws, L);
  if (!permuted) {
    if (launch_permutation(pa, ws, L, dev, s) != BEAM_OK) return BEAM_ERR_CUDA;
    record(3, s);
  }
  uint16_t* x16 = at<uint16_t>(ws, L.x_perm);
  uint16_t* h16 = at<uint16_t>(ws, L.h);
  float* y = at<float>(ws, L.y);
  beam::launch_gather_f16(static_cast<const uint16_t*>(hidden), pa.perm_src,
                          pa.offsets + c.n_experts, TK, c.topk, c.d, x16, s);
  record(4, s);
  if (cudaGetLastError() != cudaSuccess) return BEAM_ERR_CUDA;

  const int64_t EF = static_cast<int64_t>(c.n_experts) * c.d_ff;
  const int64_t ED = static_cast<int64_t>(c.n_experts) * c.d;
  CUtensorMap tm_g, tm_u, tm_d, tm_x, tm_h;
  if (!tmap_u8(&tm_g, gate.q, EF, c.d / 2, 128, 128) ||
      !tmap_u8(&tm_u, up.q, EF, c.d / 2, 128, 128) ||
      !tmap_u8(&tm_d, down.q, ED, c.d_ff / 2, 128, 128) || !tmap_bf16(&tm_x, x16, rows, c.d, nt) ||
      !tmap_bf16(&tm_h, h16, rows, c.d_ff, nt))
    return BEAM_ERR_CUDA;
  beam::W4a16GemmArgs ga{};
  ga.counts = pa.counts;
  ga.offsets = pa.offsets;
  ga.perm_w = pa.perm_w;
  ga.E = c.n_experts;
  ga.status = at<uint32_t>(ws, L.status);
  ga.wait_limit_ns = g_wait_ns;
  ga.weight_evict_first = small_batch(c, TK) ? 1 : 0;
  auto grid_for = [&](int m_blocks) {
    const int64_t tiles = static_cast<int64_t>(m_blocks) * (c.n_experts + (TK + nt - 1) / nt);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev.sms, tiles)));
  };
  ga.sfa0 = gate.sf;
  ga.sfa1 = up.sf;
  ga.gs0 = gate.global_scale;
  ga.gs1 = up.global_scale;
  ga.h_out = h16;
  ga.out_ld = c.d_ff;
  ga.rows_per_expert = c.d_ff;
  ga.m_blocks = c.d_ff / 128;
  ga.k_blocks = c.d / 256;
  ga.a_rows = static_cast<int32_t>(EF);
  ga.b_rows = static_cast<int32_t>(rows);
  ga.out_rows_cap = static_cast<int32_t>(rows);
  if (beam::launch_w4a16_gemm(true, nt, tm_g, tm_u, tm_x, ga, grid_for(ga.m_blocks), s) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  record(5, s);
  ga.sfa0 = down.sf;
  ga.sfa1 = nullptr;
  ga.gs0 = down.global_scale;
  ga.gs1 = nullptr;
  ga.h_out = nullptr;
  ga.y_out = y;
  ga.out_ld = c.d;
  ga.rows_per_expert = c.d;
  // pairs of adjacent 128-row W_d blocks share each token tile (d % 256 == 0
  // here): two weight tiles per stage, as in gate/up, keep the converters
  // and MMA issuers busy
  ga.m_blocks = c.d / 256;
  ga.k_blocks = c.d_ff / 256;
  ga.a_rows = static_cast<int32_t>(ED);
  ga.out_rows_cap = static_cast<int32_t>(rows);
  if (beam::launch_w4a16_gemm(false, nt, tm_d, tm_d, tm_h, ga, grid_for(ga.m_blocks), s) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  record(6, s);
  if (finish_combine(c, y, pa.pair_row, T, out, nullptr, boundary, pa.status, s) != cudaSuccess)
    return BEAM_ERR_CUDA;
  record(7, s);
  return cuda_status(cudaGetLastError());
}

bool valid_fp4_weight(const beam_fp4_weight_t* w) {
  return w && aligned16(w->q) && aligned16(w->sf) && aligned16(w->global_scale);
}

bool valid_fp8_weight(const beam_fp8_weight_t* w) {
  return w && aligned16(w->q) && aligned16(w->scale);
}

bool valid_mxfp8_weight(const beam_mxfp8_weight_t* w) {
  return w && aligned16(w->q) && aligned16(w->sf);
}

// The boundary's own argument checks that need no pointer (they come before
// the empty-batch return, so a bad description fails at T = 0 too): n >= 1,
// eps >= 0, and a token's FP32 values fit the combine kernel's shared memory.
bool boundary_shape_ok(const beam_moe_config_t* cfg, const beam_moe_boundary_t* b) {
  return b && b->residual_index >= 1 && b->eps >= 0.f &&
         static_cast<int64_t>(cfg->d) * 4 <= 200 * 1024;
}

// The combine kernel's boundary arguments: c_h = sqrt((n-1)/n) and
// c_x = 1/sqrt(n) in double, rounded once to FP32.  False for an unaligned
// buffer.
bool boundary_args(const beam_moe_boundary_t* b, beam::BoundaryArgs* ba) {
  if (!aligned16(b->residual) || !aligned16(b->post_norm_w) || !aligned16(b->next_norm_w) ||
      !aligned16(b->next_input))
    return false;
  ba->g_post = static_cast<const uint16_t*>(b->post_norm_w);
  ba->g_pre = static_cast<const uint16_t*>(b->next_norm_w);
  ba->residual = static_cast<uint16_t*>(b->residual);
  ba->next_x = static_cast<uint16_t*>(b->next_input);
  ba->eps = b->eps;
  const double n = b->residual_index;
  ba->c_h = static_cast<float>(std::sqrt((n - 1.0) / n));
  ba->c_x = static_cast<float>(1.0 / std::sqrt(n));
  return true;
}

// The body every quantised-expert layer call shares: checks, routing, then
// run(idx, w, layout, dev, stream, permuted, boundary) for the format's
// expert kernels.  bnd == nullptr: the plain layer.
template <class W, class Valid, class Run>
beam_status_t forward_quantised(const beam_moe_config_t* cfg, int32_t fmt, const void* hidden,
                                const float* router_w, const float* corr_bias, const W* gate,
                                const W* up, const W* down, void* out, int64_t T,
                                const beam_moe_boundary_t* bnd, void* workspace, size_t ws_bytes,
                                void* stream, Valid valid, Run run) {
  Layout L;
  DevInfo dev;
  bool empty = false;
  beam_status_t st = common_checks(cfg, T, workspace, ws_bytes, &L, &dev, &empty, fmt);
  if (st != BEAM_OK) return st;
  if (bnd && !boundary_shape_ok(cfg, bnd)) return BEAM_ERR_INVALID_ARG;
  if (empty) return BEAM_OK;
  if (!aligned16(hidden) || !aligned16(router_w) || !aligned16(corr_bias) || !valid(gate) ||
      !valid(up) || !valid(down) || !aligned16(out))
    return BEAM_ERR_INVALID_ARG;
  beam::BoundaryArgs ba;
  if (bnd && !boundary_args(bnd, &ba)) return BEAM_ERR_INVALID_ARG;
  if (!encoder()) return BEAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  record(0, s);
  int32_t* idx = at<int32_t>(workspace, L.idx);
  float* w = at<float>(workspace, L.w);
  bool permuted = false;
  st = run_route(*cfg, hidden, router_w, corr_bias, T, idx, w, at<float>(workspace, L.logits),
                 workspace, L, dev, s, &permuted);
  if (st != BEAM_OK) return st;
  return run(idx, w, L, dev, s, permuted, bnd ? &ba : nullptr);
}

// ---------------------------------------------------------------- no-allocation scratch
// Scratch for beam_moe_forward_noalloc, which serves callers that cannot
// allocate device memory.  A fixed-size device array takes the place of the
// caller's workspace.  Every GPU that loads this library's module holds it
// until the process exits.  In host code `g_noalloc_scratch` only names the
// symbol: its device address comes from cudaGetSymbolAddress, taken once per
// device with that device current.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The context current on the calling thread (the driver's cuCtxGetCurrent,
// fetched through the runtime like the tensor-map encoder); nullptr if the
// query fails.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// The array's device address on the current device, looked up once per
// device and context: a new context on the device (after cudaDeviceReset,
// say) loads the module again at another address, so the cached one is
// dropped when the current context is not the one it was taken in.
void* noalloc_scratch_address() {
  static void* addr[64] = {};
  static CUcontext ctx[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  CUcontext cur = current_context();  // none yet on a thread that has not used the device
  std::lock_guard<std::mutex> lock(mu);
  if (!cur || !addr[dev] || ctx[dev] != cur) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    cur = current_context();  // the lookup made the device's context current
    if (!cur) return nullptr;
    addr[dev] = p;
    ctx[dev] = cur;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

size_t beam_moe_workspace_size(const beam_moe_config_t* cfg, int64_t T_max, int32_t weight_fmt) {
  if (!valid_cfg(cfg) || T_max < 0 || !known_fmt(weight_fmt)) return 0;
  return make_layout(*cfg, T_max, weight_fmt).total;
}

beam_status_t beam_moe_workspace_layout(const beam_moe_config_t* cfg, int64_t T_max,
                                        int32_t weight_fmt, beam_moe_ws_layout_t* out) {
  if (!out || !valid_cfg(cfg) || T_max < 0 || !known_fmt(weight_fmt)) return BEAM_ERR_INVALID_ARG;
  const Layout L = make_layout(*cfg, T_max, weight_fmt);
  out->status = L.status;
  out->logits = L.logits;
  out->topk_idx = L.idx;
  out->topk_w = L.w;
  out->counts = L.counts;
  out->offsets = L.offsets;
  out->perm_src = L.perm_src;
  out->pair_row = L.pair_row;
  out->perm_w = L.perm_w;
  out->x_perm = L.x_perm;
  out->h = L.h;
  out->x_fp4 = L.x_fp4;
  out->x_sf = L.x_sf;
  out->h_fp4 = L.h_fp4;
  out->h_sf = L.h_sf;
  out->y = L.y;
  out->x_fp8 = L.x_fp8;
  out->x_scale = L.x_scale;
  out->h_fp8 = L.h_fp8;
  out->h_scale = L.h_scale;
  out->total = L.total;
  return BEAM_OK;
}

beam_status_t beam_moe_route(const beam_moe_config_t* cfg, const void* hidden,
                             const float* router_w, const float* corr_bias, int64_t T,
                             int32_t* topk_idx, float* topk_w, float* logits, void* workspace,
                             size_t ws_bytes, void* stream) {
  Layout L;
  DevInfo dev;
  bool empty = false;
  beam_status_t st = common_checks(cfg, T, workspace, ws_bytes, &L, &dev, &empty);
  if (st != BEAM_OK || empty) return st;
  if (!aligned16(hidden) || !aligned16(router_w) || !aligned16(corr_bias) ||
      !aligned16(topk_idx) || !aligned16(topk_w) || (logits && !aligned16(logits)))
    return BEAM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tensor_router(*cfg, T) && !encoder()) return BEAM_ERR_CUDA;
  return run_route(*cfg, hidden, router_w, corr_bias, T, topk_idx, topk_w,
                   logits ? logits : at<float>(workspace, L.logits), workspace, L, dev, s);
}

beam_status_t beam_moe_select(const beam_moe_config_t* cfg, const float* logits,
                              const float* corr_bias, int64_t T, int32_t* topk_idx, float* topk_w,
                              void* workspace, size_t ws_bytes, void* stream) {
  Layout L;
  DevInfo dev;
  bool empty = false;
  beam_status_t st = common_checks(cfg, T, workspace, ws_bytes, &L, &dev, &empty);
  if (st != BEAM_OK || empty) return st;
  if (!aligned16(logits) || !aligned16(corr_bias) || !aligned16(topk_idx) || !aligned16(topk_w))
    return BEAM_ERR_INVALID_ARG;
  beam::SelectArgs sa;
  sa.part = logits;
  sa.ksplit = 1;
  sa.bias = corr_bias;
  sa.T = T;
  sa.E = cfg->n_experts;
  sa.G = cfg->n_groups;
  sa.kg = cfg->topk_groups;
  sa.k = cfg->topk;
  sa.alpha = cfg->routed_scale;
  sa.idx = topk_idx;
  sa.w = topk_w;
  sa.logits = nullptr;
  beam::launch_select(sa, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

beam_status_t beam_moe_forward(const beam_moe_config_t* cfg, const void* hidden,
                               const float* router_w, const float* corr_bias, const void* w_gate,
                               const void* w_up, const void* w_down, void* out, int64_t T,
                               void* workspace, size_t ws_bytes, void* stream) {
  Layout L;
  DevInfo dev;
  bool empty = false;
  beam_status_t st = common_checks(cfg, T, workspace, ws_bytes, &L, &dev, &empty);
  if (st != BEAM_OK || empty) return st;
  if (!aligned16(hidden) || !aligned16(router_w) || !aligned16(corr_bias) || !aligned16(w_gate) ||
      !aligned16(w_up) || !aligned16(w_down) || !aligned16(out))
    return BEAM_ERR_INVALID_ARG;
  if (!encoder()) return BEAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  record(0, s);
  int32_t* idx = at<int32_t>(workspace, L.idx);
  float* w = at<float>(workspace, L.w);
  bool permuted = false;
  st = run_route(*cfg, hidden, router_w, corr_bias, T, idx, w, at<float>(workspace, L.logits),
                 workspace, L, dev, s, &permuted);
  if (st != BEAM_OK) return st;
  return run_experts(*cfg, hidden, idx, w, w_gate, w_up, w_down, out, T, workspace, L, dev, s,
                     permuted);
}

beam_status_t beam_moe_forward_boundary(const beam_moe_config_t* cfg, const void* hidden,
                                        const float* router_w, const float* corr_bias,
                                        const void* w_gate, const void* w_up, const void* w_down,
                                        void* out, int64_t T, const beam_moe_boundary_t* bnd,
                                        void* workspace, size_t ws_bytes, void* stream) {
  Layout L;
  DevInfo dev;
  bool empty = false;
  beam_status_t st = common_checks(cfg, T, workspace, ws_bytes, &L, &dev, &empty);
  if (st != BEAM_OK) return st;
  if (!boundary_shape_ok(cfg, bnd)) return BEAM_ERR_INVALID_ARG;
  if (empty) return BEAM_OK;
  beam::BoundaryArgs ba;
  if (!aligned16(hidden) || !aligned16(router_w) || !aligned16(corr_bias) || !aligned16(w_gate) ||
      !aligned16(w_up) || !aligned16(w_down) || !aligned16(out) || !boundary_args(bnd, &ba))
    return BEAM_ERR_INVALID_ARG;
  if (!encoder()) return BEAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  record(0, s);
  int32_t* idx = at<int32_t>(workspace, L.idx);
  float* w = at<float>(workspace, L.w);
  bool permuted = false;
  st = run_route(*cfg, hidden, router_w, corr_bias, T, idx, w, at<float>(workspace, L.logits),
                 workspace, L, dev, s, &permuted);
  if (st != BEAM_OK) return st;
  return run_experts(*cfg, hidden, idx, w, w_gate, w_up, w_down, out, T, workspace, L, dev, s,
                     permuted, nullptr, 0, &ba);
}

beam_status_t beam_moe_forward_routed(const beam_moe_config_t* cfg, const void* hidden,
                                      const int32_t* topk_idx, const float* topk_w,
                                      const void* w_gate, const void* w_up, const void* w_down,
                                      void* out, int64_t T, void* workspace, size_t ws_bytes,
                                      void* stream) {
  Layout L;
  DevInfo dev;
  bool empty = false;
  beam_status_t st = common_checks(cfg, T, workspace, ws_bytes, &L, &dev, &empty);
  if (st != BEAM_OK || empty) return st;
  if (!aligned16(hidden) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(w_gate) ||
      !aligned16(w_up) || !aligned16(w_down) || !aligned16(out))
    return BEAM_ERR_INVALID_ARG;
  if (!encoder()) return BEAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  record(0, s);
  record(1, s);
  record(2, s);
  return run_experts(*cfg, hidden, topk_idx, topk_w, w_gate, w_up, w_down, out, T, workspace, L,
                     dev, s);
}

beam_status_t beam_moe_forward_noalloc(const beam_moe_config_t* cfg, const void* hidden,
                                       const float* router_w, const float* corr_bias,
                                       const void* w_gate, const void* w_up, const void* w_down,
                                       void* out, int64_t T, void* stream) {
  if (!valid_cfg(cfg) || T < 0 || T > (int64_t(1) << 31) / 64) return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  if (make_layout(*cfg, T).total > kNoAllocScratchBytes) return BEAM_ERR_WORKSPACE;
  void* scratch = noalloc_scratch_address();
  if (!scratch) return BEAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status word latches the first kernel-side error: it must start at 0
  if (cudaMemsetAsync(scratch, 0, kAlign, s) != cudaSuccess) return BEAM_ERR_CUDA;
  return beam_moe_forward(cfg, hidden, router_w, corr_bias, w_gate, w_up, w_down, out, T,
                          scratch, kNoAllocScratchBytes, stream);
}

beam_status_t beam_moe_nvfp4_pack_scales(const uint8_t* sf_rowmajor, int64_t rows, int64_t S,
                                         uint8_t* sf_blocked, void* stream) {
  if (rows < 0 || S <= 0 || rows % 128 || S % 4) return BEAM_ERR_INVALID_ARG;
  if (rows == 0) return BEAM_OK;
  if (!aligned16(sf_rowmajor) || !aligned16(sf_blocked)) return BEAM_ERR_INVALID_ARG;
  DevInfo dev;
  if (!device_info(&dev)) return BEAM_ERR_CUDA;
  if (!dev.supported) return BEAM_ERR_UNSUPPORTED;
  beam::launch_pack_scales(sf_rowmajor, rows, S, sf_blocked, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

beam_status_t beam_moe_forward_nvfp4(const beam_moe_config_t* cfg, const void* hidden,
                                     const float* router_w, const float* corr_bias,
                                     const beam_fp4_weight_t* gate, const beam_fp4_weight_t* up,
                                     const beam_fp4_weight_t* down, void* out, int64_t T,
                                     void* workspace, size_t ws_bytes, void* stream) {
  return beam_moe_forward_nvfp4_boundary(cfg, hidden, router_w, corr_bias, gate, up, down, out, T,
                                         nullptr, workspace, ws_bytes, stream);
}

beam_status_t beam_moe_forward_nvfp4_boundary(const beam_moe_config_t* cfg, const void* hidden,
                                              const float* router_w, const float* corr_bias,
                                              const beam_fp4_weight_t* gate,
                                              const beam_fp4_weight_t* up,
                                              const beam_fp4_weight_t* down, void* out, int64_t T,
                                              const beam_moe_boundary_t* boundary,
                                              void* workspace, size_t ws_bytes, void* stream) {
  return forward_quantised(
      cfg, BEAM_WEIGHTS_NVFP4, hidden, router_w, corr_bias, gate, up, down, out, T, boundary,
      workspace, ws_bytes, stream, valid_fp4_weight,
      [&](const int32_t* idx, const float* w, const Layout& L, const DevInfo& dev,
          cudaStream_t s, bool permuted, const beam::BoundaryArgs* ba) {
        return run_experts_nvfp4(*cfg, hidden, idx, w, *gate, *up, *down, out, T, workspace, L,
                                 dev, s, permuted, nullptr, 0, ba);
      });
}

beam_status_t beam_moe_forward_fp8(const beam_moe_config_t* cfg, const void* hidden,
                                   const float* router_w, const float* corr_bias,
                                   const beam_fp8_weight_t* gate, const beam_fp8_weight_t* up,
                                   const beam_fp8_weight_t* down, void* out, int64_t T,
                                   void* workspace, size_t ws_bytes, void* stream) {
  return beam_moe_forward_fp8_boundary(cfg, hidden, router_w, corr_bias, gate, up, down, out, T,
                                       nullptr, workspace, ws_bytes, stream);
}

beam_status_t beam_moe_forward_fp8_boundary(const beam_moe_config_t* cfg, const void* hidden,
                                            const float* router_w, const float* corr_bias,
                                            const beam_fp8_weight_t* gate,
                                            const beam_fp8_weight_t* up,
                                            const beam_fp8_weight_t* down, void* out, int64_t T,
                                            const beam_moe_boundary_t* boundary, void* workspace,
                                            size_t ws_bytes, void* stream) {
  return forward_quantised(
      cfg, BEAM_WEIGHTS_FP8, hidden, router_w, corr_bias, gate, up, down, out, T, boundary,
      workspace, ws_bytes, stream, valid_fp8_weight,
      [&](const int32_t* idx, const float* w, const Layout& L, const DevInfo& dev,
          cudaStream_t s, bool permuted, const beam::BoundaryArgs* ba) {
        return run_experts_fp8(*cfg, hidden, idx, w, *gate, *up, *down, out, T, workspace, L, dev,
                               s, permuted, nullptr, 0, ba);
      });
}

beam_status_t beam_moe_forward_mxfp8(const beam_moe_config_t* cfg, const void* hidden,
                                     const float* router_w, const float* corr_bias,
                                     const beam_mxfp8_weight_t* gate,
                                     const beam_mxfp8_weight_t* up,
                                     const beam_mxfp8_weight_t* down, void* out, int64_t T,
                                     void* workspace, size_t ws_bytes, void* stream) {
  return beam_moe_forward_mxfp8_boundary(cfg, hidden, router_w, corr_bias, gate, up, down, out, T,
                                         nullptr, workspace, ws_bytes, stream);
}

beam_status_t beam_moe_forward_mxfp8_boundary(const beam_moe_config_t* cfg, const void* hidden,
                                              const float* router_w, const float* corr_bias,
                                              const beam_mxfp8_weight_t* gate,
                                              const beam_mxfp8_weight_t* up,
                                              const beam_mxfp8_weight_t* down, void* out,
                                              int64_t T, const beam_moe_boundary_t* boundary,
                                              void* workspace, size_t ws_bytes, void* stream) {
  return forward_quantised(
      cfg, BEAM_WEIGHTS_MXFP8, hidden, router_w, corr_bias, gate, up, down, out, T, boundary,
      workspace, ws_bytes, stream, valid_mxfp8_weight,
      [&](const int32_t* idx, const float* w, const Layout& L, const DevInfo& dev,
          cudaStream_t s, bool permuted, const beam::BoundaryArgs* ba) {
        return run_experts_mxfp8(*cfg, hidden, idx, w, *gate, *up, *down, out, T, workspace, L,
                                 dev, s, permuted, ba);
      });
}

beam_status_t beam_moe_fp8_quantize_rows(const void* x, int64_t n, int32_t cols, uint8_t* q,
                                         float* scale, void* stream) {
  if (n < 0 || n > INT32_MAX || cols <= 0 || cols % 8) return BEAM_ERR_INVALID_ARG;
  if (n == 0) return BEAM_OK;
  if (!aligned16(x) || !aligned16(q) || !aligned16(scale)) return BEAM_ERR_INVALID_ARG;
  beam::launch_quantize_e4m3_rows(static_cast<const uint16_t*>(x), nullptr, n, cols, q, scale,
                                  static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

beam_status_t beam_moe_forward_nvfp4_a16(const beam_moe_config_t* cfg, const void* hidden,
                                         const float* router_w, const float* corr_bias,
                                         const beam_fp4_weight_t* gate, const beam_fp4_weight_t* up,
                                         const beam_fp4_weight_t* down, void* out, int64_t T,
                                         void* workspace, size_t ws_bytes, void* stream) {
  return beam_moe_forward_nvfp4_a16_boundary(cfg, hidden, router_w, corr_bias, gate, up, down,
                                             out, T, nullptr, workspace, ws_bytes, stream);
}

beam_status_t beam_moe_forward_nvfp4_a16_boundary(const beam_moe_config_t* cfg,
                                                  const void* hidden, const float* router_w,
                                                  const float* corr_bias,
                                                  const beam_fp4_weight_t* gate,
                                                  const beam_fp4_weight_t* up,
                                                  const beam_fp4_weight_t* down, void* out,
                                                  int64_t T, const beam_moe_boundary_t* boundary,
                                                  void* workspace, size_t ws_bytes, void* stream) {
  return forward_quantised(
      cfg, BEAM_WEIGHTS_NVFP4_A16, hidden, router_w, corr_bias, gate, up, down, out, T, boundary,
      workspace, ws_bytes, stream, valid_fp4_weight,
      [&](const int32_t* idx, const float* w, const Layout& L, const DevInfo& dev,
          cudaStream_t s, bool permuted, const beam::BoundaryArgs* ba) {
        return run_experts_w4a16(*cfg, hidden, idx, w, *gate, *up, *down, out, T, workspace, L,
                                 dev, s, permuted, ba);
      });
}

// ------------------------------------------------------- expert parallelism
namespace {

bool valid_ep(const beam_moe_config_t* c, int32_t n_ranks) {
  return valid_cfg(c) && n_ranks >= 1 && n_ranks <= c->n_experts && c->n_experts % n_ranks == 0;
}

// the expert computation of one rank: its E / n_ranks experts, one row per
// received (token, slot) pair
beam_moe_config_t local_cfg(const beam_moe_config_t& c, int32_t n_ranks) {
  beam_moe_config_t l = c;
  l.n_experts = c.n_experts / n_ranks;
  l.n_groups = 1;
  l.topk_groups = 1;
  l.topk = 1;
  return l;
}

}  // namespace

beam_status_t beam_moe_ep_dispatch(const beam_moe_config_t* cfg, const void* hidden,
                                   const float* router_w, const float* corr_bias, int64_t T,
                                   int32_t n_ranks, void* send_x, int32_t* send_expert,
                                   float* send_w, int32_t* send_counts, void* workspace,
                                   size_t ws_bytes, void* stream) {
  if (!valid_ep(cfg, n_ranks) || !aligned16(send_counts)) return BEAM_ERR_INVALID_ARG;
  Layout L;
  DevInfo dev;
  bool empty = false;
  beam_status_t st = common_checks(cfg, T, workspace, ws_bytes, &L, &dev, &empty);
  if (st != BEAM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (empty)  // a rank without tokens still reports its (zero) counts
    return cuda_status(cudaMemsetAsync(send_counts, 0, sizeof(int32_t) * n_ranks, s));
  if (!aligned16(hidden) || !aligned16(router_w) || !aligned16(corr_bias) || !aligned16(send_x) ||
      !aligned16(send_expert) || !aligned16(send_w))
    return BEAM_ERR_INVALID_ARG;
  if (!encoder()) return BEAM_ERR_CUDA;
  record(0, s);
  int32_t* idx = at<int32_t>(workspace, L.idx);
  float* w = at<float>(workspace, L.w);
  bool permuted = false;
  st = run_route(*cfg, hidden, router_w, corr_bias, T, idx, w, at<float>(workspace, L.logits),
                 workspace, L, dev, s, &permuted);
  if (st != BEAM_OK) return st;
  const beam::PermuteArgs pa = permute_args(*cfg, idx, w, T, workspace, L);
  if (!permuted && launch_permutation(pa, workspace, L, dev, s) != BEAM_OK) return BEAM_ERR_CUDA;
  record(3, s);
  const int64_t TK = T * cfg->topk;
  beam::launch_gather(static_cast<const uint16_t*>(hidden), pa.perm_src, pa.offsets + cfg->n_experts,
                      TK, cfg->topk, cfg->d, static_cast<uint16_t*>(send_x), s);
  beam::launch_ep_pack(idx, pa.perm_src, pa.perm_w, pa.offsets, TK, cfg->n_experts, n_ranks,
                       send_expert, send_w, send_counts, s);
  record(4, s);
  return cuda_status(cudaGetLastError());
}

size_t beam_moe_ep_workspace_size(const beam_moe_config_t* cfg, int32_t n_ranks, int64_t M_max,
                                  int32_t weight_fmt) {
  if (!valid_ep(cfg, n_ranks) || M_max < 0 || M_max > (int64_t(1) << 31) / 64) return 0;
  if (weight_fmt != BEAM_WEIGHTS_BF16 && weight_fmt != BEAM_WEIGHTS_NVFP4 &&
      weight_fmt != BEAM_WEIGHTS_FP8)
    return 0;
  if (weight_fmt == BEAM_WEIGHTS_NVFP4 && (cfg->d % 256 || cfg->d_ff % 256)) return 0;
  return make_layout(local_cfg(*cfg, n_ranks), std::max<int64_t>(M_max, 1), weight_fmt).total;
}

beam_status_t beam_moe_ep_experts(const beam_moe_config_t* cfg, int32_t n_ranks, int32_t rank,
                                  const void* x_recv, const int32_t* expert_recv,
                                  const float* w_recv, const void* w_gate, const void* w_up,
                                  const void* w_down, float* y_recv, int64_t M, void* workspace,
                                  size_t ws_bytes, void* stream) {
  if (!valid_ep(cfg, n_ranks) || rank < 0 || rank >= n_ranks || M < 0 ||
      M > (int64_t(1) << 31) / 64)
    return BEAM_ERR_INVALID_ARG;
  if (M == 0) return BEAM_OK;
  const beam_moe_config_t lc = local_cfg(*cfg, n_ranks);
  if (!aligned16(workspace) || !aligned16(x_recv) || !aligned16(expert_recv) ||
      !aligned16(w_recv) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(y_recv))
    return BEAM_ERR_INVALID_ARG;
  const Layout L = make_layout(lc, M);
  if (ws_bytes < L.total) return BEAM_ERR_WORKSPACE;
  DevInfo dev;
  if (!device_info(&dev)) return BEAM_ERR_CUDA;
  if (!dev.supported) return BEAM_ERR_UNSUPPORTED;
  if (!encoder()) return BEAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  record(0, s);
  record(1, s);
  record(2, s);
  return run_experts(lc, x_recv, expert_recv, w_recv, w_gate, w_up, w_down, nullptr, M, workspace,
                     L, dev, s, false, y_recv, rank * lc.n_experts);
}

beam_status_t beam_moe_ep_experts_nvfp4(const beam_moe_config_t* cfg, int32_t n_ranks,
                                        int32_t rank, const void* x_recv,
                                        const int32_t* expert_recv, const float* w_recv,
                                        const beam_fp4_weight_t* gate, const beam_fp4_weight_t* up,
                                        const beam_fp4_weight_t* down, float* y_recv, int64_t M,
                                        void* workspace, size_t ws_bytes, void* stream) {
  if (!valid_ep(cfg, n_ranks) || rank < 0 || rank >= n_ranks || M < 0 ||
      M > (int64_t(1) << 31) / 64 || cfg->d % 256 || cfg->d_ff % 256)
    return BEAM_ERR_INVALID_ARG;
  if (M == 0) return BEAM_OK;
  const beam_moe_config_t lc = local_cfg(*cfg, n_ranks);
  if (!aligned16(workspace) || !aligned16(x_recv) || !aligned16(expert_recv) ||
      !aligned16(w_recv) || !valid_fp4_weight(gate) || !valid_fp4_weight(up) ||
      !valid_fp4_weight(down) || !aligned16(y_recv))
    return BEAM_ERR_INVALID_ARG;
  const Layout L = make_layout(lc, M, BEAM_WEIGHTS_NVFP4);
  if (ws_bytes < L.total) return BEAM_ERR_WORKSPACE;
  DevInfo dev;
  if (!device_info(&dev)) return BEAM_ERR_CUDA;
  if (!dev.supported) return BEAM_ERR_UNSUPPORTED;
  if (!encoder()) return BEAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  record(0, s);
  record(1, s);
  record(2, s);
  return run_experts_nvfp4(lc, x_recv, expert_recv, w_recv, *gate, *up, *down, nullptr, M,
                           workspace, L, dev, s, false, y_recv, rank * lc.n_experts);
}

beam_status_t beam_moe_ep_experts_fp8(const beam_moe_config_t* cfg, int32_t n_ranks, int32_t rank,
                                      const void* x_recv, const int32_t* expert_recv,
                                      const float* w_recv, const beam_fp8_weight_t* gate,
                                      const beam_fp8_weight_t* up, const beam_fp8_weight_t* down,
                                      float* y_recv, int64_t M, void* workspace, size_t ws_bytes,
                                      void* stream) {
  if (!valid_ep(cfg, n_ranks) || rank < 0 || rank >= n_ranks || M < 0 ||
      M > (int64_t(1) << 31) / 64)
    return BEAM_ERR_INVALID_ARG;
  if (M == 0) return BEAM_OK;
  const beam_moe_config_t lc = local_cfg(*cfg, n_ranks);
  if (!aligned16(workspace) || !aligned16(x_recv) || !aligned16(expert_recv) ||
      !aligned16(w_recv) || !valid_fp8_weight(gate) || !valid_fp8_weight(up) ||
      !valid_fp8_weight(down) || !aligned16(y_recv))
    return BEAM_ERR_INVALID_ARG;
  const Layout L = make_layout(lc, M, BEAM_WEIGHTS_FP8);
  if (ws_bytes < L.total) return BEAM_ERR_WORKSPACE;
  DevInfo dev;
  if (!device_info(&dev)) return BEAM_ERR_CUDA;
  if (!dev.supported) return BEAM_ERR_UNSUPPORTED;
  if (!encoder()) return BEAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  record(0, s);
  record(1, s);
  record(2, s);
  // one received row per (token, slot): the rows are quantised per row, which
  // gives each the codes and scale of its token
  return run_experts_fp8(lc, x_recv, expert_recv, w_recv, *gate, *up, *down, nullptr, M,
                         workspace, L, dev, s, false, y_recv, rank * lc.n_experts);
}

beam_status_t beam_moe_ep_combine(const beam_moe_config_t* cfg, const float* y_back, int64_t T,
                                  void* out, void* workspace, size_t ws_bytes, void* stream) {
  Layout L;
  DevInfo dev;
  bool empty = false;
  beam_status_t st = common_checks(cfg, T, workspace, ws_bytes, &L, &dev, &empty);
  if (st != BEAM_OK || empty) return st;
  if (!aligned16(y_back) || !aligned16(out)) return BEAM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  beam::launch_combine(y_back, at<int32_t>(workspace, L.pair_row), T, cfg->topk, cfg->d,
                       static_cast<uint16_t*>(out), at<uint32_t>(workspace, L.status), s);
  record(7, s);
  return cuda_status(cudaGetLastError());
}

beam_status_t beam_moe_check_status(void* workspace, void* stream) {
  if (!aligned16(workspace)) return BEAM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BEAM_ERR_CUDA;
  // the status word sits at offset 0 of every layout
  if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return BEAM_ERR_CUDA;
  if (v != 0 && cudaMemset(workspace, 0, sizeof v) != cudaSuccess) return BEAM_ERR_CUDA;
  return static_cast<beam_status_t>(v);
}

beam_status_t beam_moe_set_stage_events(void* const* events, int32_t n) {
  if (n == 0) {
    g_num_events = 0;
    return BEAM_OK;
  }
  if (!events || n < 8) return BEAM_ERR_INVALID_ARG;
  for (int i = 0; i < 8; ++i) {
    if (!events[i]) return BEAM_ERR_INVALID_ARG;
    g_events[i] = static_cast<cudaEvent_t>(events[i]);
  }
  g_num_events = 8;
  return BEAM_OK;
}

beam_status_t beam_moe_set_debug(uint32_t wait_limit_us, int32_t withhold_first_load) {
  g_wait_ns = wait_limit_us ? static_cast<uint64_t>(wait_limit_us) * 1000ull : kDefaultWaitNs;
  g_withhold = withhold_first_load ? 1 : 0;
  return BEAM_OK;
}

int32_t beam_moe_kernels_per_forward(const beam_moe_config_t* cfg, int64_t T, int32_t weight_fmt,
                                     int32_t routed) {
  if (!valid_cfg(cfg) || T <= 0 || !known_fmt(weight_fmt)) return 0;
  if (routed && weight_fmt != BEAM_WEIGHTS_BF16) return 0;
  // experts: permute, gather (BF16, larger batches) or row quantisation
  // (NVFP4) or F16 gather (W4A16), gate/up, down, combine; FP8 quantises the
  // token rows and h (and gathers the token codes for larger batches)
  const bool small = small_batch(*cfg, T * cfg->topk);
  const int experts = weight_fmt == BEAM_WEIGHTS_FP8    ? 6 + (small ? 0 : 1)
                      : weight_fmt != BEAM_WEIGHTS_BF16 ? 5  // NVFP4, W4A16, MXFP8
                                                        : 4 + (small ? 0 : 1);
  if (routed) return experts;
  // routing: router (+ plane split), select; decode-sized batches run router,
  // select and permute as one launch
  return experts + 2 + (tensor_router(*cfg, T) ? 1 : 0) - (fused_routing(*cfg, T) ? 2 : 0);
}

const char* beam_status_string(beam_status_t s) {
  switch (s) {
    case BEAM_OK: return "ok";
    case BEAM_ERR_INVALID_ARG: return "invalid argument";
    case BEAM_ERR_UNSUPPORTED: return "unsupported (needs an sm_103 GPU)";
    case BEAM_ERR_WORKSPACE: return "workspace too small";
    case BEAM_ERR_CUDA: return "CUDA error";
    case BEAM_ERR_TIMEOUT: return "device-side wait timed out";
    case BEAM_ERR_DEVICE_CHECK: return "device-side argument check failed";
  }
  return "unknown status";
}

}  // extern "C"
