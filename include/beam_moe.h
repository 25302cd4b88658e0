/*
 * beam_moe.h -- C ABI of the Beam MoE layer for NVIDIA GB300 (sm_103a).
 *
 * The layer is the sparse feed-forward block of the Beam 501B-A23B model:
 *   1. an FP32 router, logits = x W_r^T
 *      ("SGLang 原生支持 Reflection 的 Beam 并驱动其生产 API", section "Dense
 *      Layers and Grouped MoE Routing"; "vLLM 实现 Reflection Beam 501B MoE
 *      模型 Day 0 支持", section "MoE and residual stream": router weights,
 *      accumulation and logits all FP32);
 *   2. DeepSeek-V3-style group-limited selection: sigmoid scores s plus a
 *      correction bias b give choice scores c = s + b; groups are ranked by the
 *      sum of their two best c; the best topk_groups groups are kept; the topk
 *      best experts of the kept groups are chosen; their s are renormalised
 *      and multiplied by routed_scale (vLLM post, same section; "Reflection
 *      发布 501B 开源模型 Beam，Apache 2.0 许可", section "专家混合");
 *   3. SwiGLU experts h = silu(x W_g^T) * (x W_u^T) with the product in FP32,
 *      rounded to BF16, then y = h W_d^T (HF post, sections "专家混合" and
 *      "残差流"; SGLang post, section "BF16 MoE Kernel Optimization");
 *   4. the weighted combine out = bf16(sum_k w_k y_k): FP32 routing weights
 *      applied to FP32 expert outputs, summed locally in FP32 in slot order
 *      and rounded once to BF16 (SGLang post, sections "BF16 MoE Kernel
 *      Optimization" and "Fusion Optimizations").
 *   There is no shared expert.
 *
 * Conventions shared by every entry point
 *   - Every pointer except `stream` is DEVICE memory on the current device,
 *     allocated and owned by the caller; the library never frees or keeps it
 *     past the call and allocates no device memory of its own.
 *   - Row-major layouts, nn.Linear weight convention ([out, in], K contiguous):
 *       hidden   [T, d]      BF16
 *       router_w [E, d]      FP32
 *       corr_bias[E]         FP32
 *       w_gate   [E, F, d]   BF16      (F = d_ff)
 *       w_up     [E, F, d]   BF16
 *       w_down   [E, d, F]   BF16
 *       out      [T, d]      BF16
 *       topk_idx [T, topk]   int32, slots in descending choice score
 *       topk_w   [T, topk]   FP32, includes routed_scale (sums to it)
 *   - Pointers must be 16-byte aligned.  Shapes: d % 128 == 0,
 *     d_ff % 128 == 0, n_experts % 32 == 0 and <= 256, n_groups divides
 *     n_experts with 2 <= n_experts/n_groups <= 32 a power of two,
 *     1 <= topk_groups <= n_groups, 1 <= topk <= min(32, topk_groups *
 *     n_experts / n_groups), T >= 0.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  No entry point synchronises or copies between host
 *     and device, except beam_moe_check_status.  Kernels after a call's
 *     first one are launched with programmatic stream serialization (SGLang
 *     post, "Fusion Optimizations"): each may start before the kernel ahead
 *     of it on the stream has finished, and waits on the device
 *     (griddepcontrol.wait) before it reads anything that kernel writes, so
 *     the order against the caller's own work on the stream is that of
 *     ordinary launches.  A caller's kernel launched after a call with the
 *     same attribute may likewise start early, and must wait the same way
 *     before it reads the call's outputs.
 *   - Every entry point returns a status and never aborts or prints.  Invalid
 *     arguments are rejected before anything is launched (outputs untouched).
 *     T == 0 with a valid cfg returns BEAM_OK at once: nothing is launched
 *     and no pointer is looked at.  Errors found by the kernels
 *     (a wait that ran out of time, an expert index out of range) are latched
 *     in the workspace's status word and reported by beam_moe_check_status.
 *   - Results are deterministic: no floating-point atomics; every reduction
 *     runs in a fixed order.
 */
#ifndef BEAM_MOE_H_
#define BEAM_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BEAM_OK = 0,
  BEAM_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape, T < 0   */
  BEAM_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. no sm_103)  */
  BEAM_ERR_WORKSPACE = 3,     /* workspace smaller than beam_moe_workspace_size */
  BEAM_ERR_CUDA = 4,          /* a CUDA call or launch failed                */
  BEAM_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out          */
  BEAM_ERR_DEVICE_CHECK = 6   /* a device-side argument check failed         */
} beam_status_t;

/* Layer shape.  Beam: {5120, 256, 8, 4, 8, 2560, 2.5f}. */
typedef struct {
  int32_t d;             /* hidden size                                   */
  int32_t n_experts;     /* routed experts E                              */
  int32_t n_groups;      /* expert groups G                               */
  int32_t topk_groups;   /* groups kept per token                         */
  int32_t topk;          /* experts chosen per token                      */
  int32_t d_ff;          /* expert intermediate size F                    */
  float routed_scale;    /* factor on the renormalised weights (2.5)      */
} beam_moe_config_t;

/* Weight formats for beam_moe_workspace_size. */
#define BEAM_WEIGHTS_BF16 0
#define BEAM_WEIGHTS_NVFP4 1
#define BEAM_WEIGHTS_NVFP4_A16 2 /* NVFP4 weights, 16-bit activations */
#define BEAM_WEIGHTS_FP8 3       /* dynamic FP8: E4M3 weights and activations */
#define BEAM_WEIGHTS_MXFP8 4     /* MXFP8: E4M3 with E8M0 scales per 32, weights and activations */

/* Bytes of device workspace a call with up to T_max tokens needs (256-byte
 * aligned).  Returns 0 for an invalid configuration. */
size_t beam_moe_workspace_size(const beam_moe_config_t *cfg, int64_t T_max,
                               int32_t weight_fmt);

/* Byte offsets of the intermediate buffers inside the workspace (for
 * inspection in tests and tools; the layout depends on cfg and T_max).
 * perm_* arrays are indexed by "permuted row": the (token, slot) pairs sorted
 * stably by expert, then token, then slot. */
typedef struct {
  size_t status;        /* uint32 status word (BEAM_OK or the first error)   */
  size_t logits;        /* FP32 [T, E] (router output as the selection read it) */
  size_t topk_idx;      /* int32 [T, topk]                                    */
  size_t topk_w;        /* FP32 [T, topk]                                     */
  size_t counts;        /* int32 [E] rows per expert                          */
  size_t offsets;       /* int32 [E + 1] first permuted row of each expert    */
  size_t perm_src;      /* int32 [T*topk] permuted row -> token*topk + slot   */
  size_t pair_row;      /* int32 [T*topk] token*topk + slot -> permuted row   */
  size_t perm_w;        /* FP32 [T*topk] routing weight of each permuted row  */
  size_t x_perm;        /* BF16 [T*topk, d] gathered expert inputs (only when
                           T*topk > 4*E; smaller batches gather in the GEMM) */
  size_t h;             /* BF16 [T*topk, F] SwiGLU activations                */
  size_t x_fp4;         /* NVFP4 path: token rows, E2M1 codes [T*topk, d/2]   */
  size_t x_sf;          /*   their E4M3 scales [T*topk, d/4]: per 64 elements a
                             16-byte slot, 4 scales then padding             */
  size_t h_fp4;         /*   SwiGLU activations [T*topk, F/2]                  */
  size_t h_sf;          /*   and their scales [T*topk, F/4], same slots        */
                        /* MXFP8 path: the same four buffers hold E4M3 codes
                           [T*topk, d] and [T*topk, F] and E8M0 scales
                           [T*topk, d/8] and [T*topk, F/8] (per 128 elements
                           a 16-byte slot, 4 scales then padding)            */
  size_t y;             /* FP32 [T*topk, d] weighted expert outputs           */
  size_t x_fp8;         /* FP8 path: token rows, E4M3 codes [T, d]            */
  size_t x_scale;       /*   their FP32 scales [T]                            */
  size_t h_fp8;         /*   SwiGLU activations, E4M3 codes [T*topk, F] (x_perm
                             holds the gathered token codes [T*topk, d] when
                             T*topk > 4*E)                                   */
  size_t h_scale;       /*   their FP32 scales [T*topk]                       */
  size_t total;         /* == beam_moe_workspace_size                         */
} beam_moe_ws_layout_t;

beam_status_t beam_moe_workspace_layout(const beam_moe_config_t *cfg, int64_t T_max,
                                        int32_t weight_fmt, beam_moe_ws_layout_t *out);

/* Steps 1-2 only (router + group-limited selection), e.g. to record routes
 * for routing replay (SGLang post, section "Reinforcement learning in Miles":
 * recorded expert choices reused instead of recomputing top-k).
 * Writes topk_idx [T, topk], topk_w [T, topk] and, when `logits` is not
 * NULL, the FP32 router logits [T, E]. */
beam_status_t beam_moe_route(const beam_moe_config_t *cfg, const void *hidden,
                             const float *router_w, const float *corr_bias, int64_t T,
                             int32_t *topk_idx, float *topk_w, float *logits,
                             void *workspace, size_t ws_bytes, void *stream);

/* Step 2 alone on given FP32 logits [T, E] (selection tested in isolation). */
beam_status_t beam_moe_select(const beam_moe_config_t *cfg, const float *logits,
                              const float *corr_bias, int64_t T, int32_t *topk_idx,
                              float *topk_w, void *workspace, size_t ws_bytes,
                              void *stream);

/* The whole layer, steps 1-4: out [T, d] BF16. */
beam_status_t beam_moe_forward(const beam_moe_config_t *cfg, const void *hidden,
                               const float *router_w, const float *corr_bias,
                               const void *w_gate, const void *w_up, const void *w_down,
                               void *out, int64_t T, void *workspace, size_t ws_bytes,
                               void *stream);

/* Steps 3-4 with a given routing (topk_idx/topk_w as beam_moe_route writes
 * them; routing replay).  Indices outside [0, E) latch
 * BEAM_ERR_DEVICE_CHECK and contribute nothing. */
beam_status_t beam_moe_forward_routed(const beam_moe_config_t *cfg, const void *hidden,
                                      const int32_t *topk_idx, const float *topk_w,
                                      const void *w_gate, const void *w_up,
                                      const void *w_down, void *out, int64_t T,
                                      void *workspace, size_t ws_bytes, void *stream);

/* The decoder's sublayer boundary after this layer ("vLLM 实现 Reflection Beam
 * 501B MoE 模型 Day 0 支持", section "MoE and residual stream": sandwich norm and
 * depth-scaled residuals; section "Agent-driven optimization", items 1 and 3:
 * post-norm, scaled residual add and next pre-norm as one kernel that also
 * combines the top-8 expert outputs; "SGLang 原生支持 Reflection 的 Beam 并驱动其
 * 生产 API", section "Sandwich Normalization and Depth-Scaled Residuals": both
 * scaled operands are rounded to BF16 before the addition).  All device
 * pointers, BF16, 16-byte aligned, caller-owned. */
typedef struct {
  void *residual;          /* [T, d] the residual stream h; overwritten with h'     */
  const void *post_norm_w; /* [d] RMSNorm weight after the MoE sublayer           */
  const void *next_norm_w; /* [d] RMSNorm weight before the next sublayer         */
  void *next_input;        /* [T, d] out: the next sublayer's normalised input    */
  float eps;               /* RMSNorm epsilon (>= 0)                              */
  int32_t residual_index;  /* n >= 1: this is the decoder's n-th residual add     */
} beam_moe_boundary_t;

/* beam_moe_forward (out = the layer's BF16 output m, as there) followed, in
 * the combine kernel, by the boundary, per token in FP32 arithmetic:
 *   p  = bf16(m * post_norm_w / sqrt(mean(m^2) + eps))
 *   h' = bf16(bf16(c_h * h) + bf16(c_x * p)),  c_h = fp32(sqrt((n-1)/n)),
 *                                                c_x = fp32(1/sqrt(n))
 *   next_input = bf16(h' * next_norm_w / sqrt(mean(h'^2) + eps))
 * Deterministic (fixed-order sums).  BEAM_ERR_INVALID_ARG for n < 1, eps < 0
 * or d > 51200 (the token's values are staged in shared memory). */
beam_status_t beam_moe_forward_boundary(const beam_moe_config_t *cfg, const void *hidden,
                                        const float *router_w, const float *corr_bias,
                                        const void *w_gate, const void *w_up, const void *w_down,
                                        void *out, int64_t T, const beam_moe_boundary_t *boundary,
                                        void *workspace, size_t ws_bytes, void *stream);

/* beam_moe_forward without a caller workspace and without any allocation.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory at all -- a plugin inside a host application
 * that owns the whole device-memory budget and forbids allocations, or code
 * that must never enter cudaMalloc's implicit device synchronisation.  They
 * still pass every input and the output as device pointers, as for
 * beam_moe_forward; the intermediate buffers live in one fixed 32 MiB device
 * array inside this library (held on every GPU that loads the library until
 * the process exits).
 *   - Size limit: calls whose beam_moe_workspace_size(cfg, T, BEAM_WEIGHTS_BF16)
 *     exceeds 32 MiB return BEAM_ERR_WORKSPACE before anything is launched
 *     (Beam shapes: up to 128 tokens).
 *   - The first call on a device looks up the array's device address (one
 *     cudaGetSymbolAddress with that device current); make that first call
 *     before any stream capture.  The address is kept per device and
 *     context: a call in a new context on the device (after
 *     cudaDeviceReset, for instance) looks it up again.  (The other
 *     entry points' once-per-device kernel set-up is not redone after a
 *     device reset: their calls then fail with BEAM_ERR_CUDA.)
 *   - Every call shares the one array and it keeps the previous call's
 *     contents; the call clears the status word it needs at zero.  Calls
 *     whose work overlaps on the GPU (other streams, other host threads) race
 *     on it: serialise them.
 *   - Kernel-side errors latch in that private array; the return value
 *     reports argument and launch errors only.
 *   - No cudaMalloc, cudaFree or allocating library routine is called. */
beam_status_t beam_moe_forward_noalloc(const beam_moe_config_t *cfg, const void *hidden,
                                       const float *router_w, const float *corr_bias,
                                       const void *w_gate, const void *w_up,
                                       const void *w_down, void *out, int64_t T,
                                       void *stream);

/* NVFP4 expert weights of one projection (gate, up or down), N output rows
 * and K inputs per expert ("ModelOpt NVFP4" checkpoints, SGLang post, section
 * "Highlights"; vLLM post, "MoE and residual stream": NVFP4 experts).
 * A weight is q * sf * global_scale[e]. */
typedef struct {
  const uint8_t *q;             /* E2M1 codes [E, N, K/2], two per byte, low nibble = even k */
  const uint8_t *sf;            /* E4M3 scales, one per 16 along K, of the [E*N, K/16]
                                   row-major matrix in the blocked order that
                                   beam_moe_nvfp4_pack_scales writes             */
  const float *global_scale;    /* [E] FP32                                        */
} beam_fp4_weight_t;

/* Reorders row-major block scales [rows, S] (E4M3 for NVFP4, E8M0 for MXFP8;
 * rows % 128 == 0, S % 4 == 0) into blocks of 128 rows x 4 scales, 512 bytes each, block
 * (row/128, s/4) at ((row/128) * (S/4) + s/4) * 512 and byte
 * (r % 32) * 16 + (r / 32) * 4 + s % 4 inside it (r = row % 128): the order in
 * which the tensor cores take weight scales.  Run once per weight tensor when
 * the weights are loaded; `dst` is a device buffer of rows * S bytes.  No
 * counterpart on the pages (the storage order is this library's). */
beam_status_t beam_moe_nvfp4_pack_scales(const uint8_t *sf_rowmajor, int64_t rows, int64_t S,
                                         uint8_t *sf_blocked, void *stream);

/* The whole layer with NVFP4 experts.  Router and selection as in
 * beam_moe_forward; both expert GEMM inputs are quantised to NVFP4 (per 16
 * elements: scale = E4M3(amax / 6), codes = E2M1(value / scale), round to
 * nearest even, saturating; global scale 1) -- x along d before the gate/up
 * GEMM, the FP32 SwiGLU product along d_ff before the down GEMM -- and the
 * GEMMs run as block-scaled FP4 MMAs with FP32 accumulation; the per-expert
 * FP32 scales multiply the accumulators.  Extra shape rules: d % 256 == 0,
 * d_ff % 256 == 0.  Workspace: beam_moe_workspace_size(cfg, T, BEAM_WEIGHTS_NVFP4). */
beam_status_t beam_moe_forward_nvfp4(const beam_moe_config_t *cfg, const void *hidden,
                                     const float *router_w, const float *corr_bias,
                                     const beam_fp4_weight_t *gate, const beam_fp4_weight_t *up,
                                     const beam_fp4_weight_t *down, void *out, int64_t T,
                                     void *workspace, size_t ws_bytes, void *stream);

/* The whole layer with the same NVFP4 expert weights and unquantised 16-bit
 * activations (W4A16).  The tensor cores take F16 operands: each weight is
 * E2M1 code x E4M3 scale, exact in F16 (expanded in registers and stored into
 * tensor memory), times the FP32 expert scale in the epilogue; the token
 * rows are converted from BF16 to F16 (exact inside F16's normal range), and
 * the FP32 SwiGLU product is rounded to F16 for the down GEMM; magnitudes
 * beyond 65504 saturate.  Otherwise as beam_moe_forward_nvfp4 (d % 256 == 0,
 * d_ff % 256 == 0).  Workspace: beam_moe_workspace_size(cfg, T,
 * BEAM_WEIGHTS_NVFP4_A16). */
beam_status_t beam_moe_forward_nvfp4_a16(const beam_moe_config_t *cfg, const void *hidden,
                                         const float *router_w, const float *corr_bias,
                                         const beam_fp4_weight_t *gate, const beam_fp4_weight_t *up,
                                         const beam_fp4_weight_t *down, void *out, int64_t T,
                                         void *workspace, size_t ws_bytes, void *stream);

/* Dynamic FP8 expert weights (one projection of all experts): E4M3 codes
 * q [E, N, K] (K contiguous; N = d_ff for gate/up, d for down) and one FP32
 * scale per output row, scale [E, N]: the weight is code x scale (the
 * per-channel FP8 weights of a compressed-tensors dynamic FP8 checkpoint;
 * SGLang post, sections "Highlights" and "BF16, NVFP4 and FP8 Model
 * Support"). */
typedef struct {
  const uint8_t *q;     /* E4M3 [E, N, K]                                      */
  const float *scale;   /* FP32 [E, N]                                         */
} beam_fp8_weight_t;

/* The whole layer with dynamic FP8 experts.  Router and selection as in
 * beam_moe_forward.  Both expert GEMM inputs are quantised per row at run
 * time: x per token along d, and h (the FP32 SwiGLU product rounded to BF16,
 * as in beam_moe_forward) per (token, expert) row along d_ff.  The rule:
 * scale = amax / 448 in FP32 (1 for an all-zero row), code = E4M3(value /
 * scale) with an FP32 division, round to nearest even, saturating at 448.
 * The GEMMs run as E4M3 x E4M3 tensor-core MMAs with FP32 accumulation; the
 * weight row's and the token row's scales multiply each accumulator; the
 * rest (FP32 routing weights, FP32 combine in slot order, one BF16 rounding)
 * is beam_moe_forward's.  Workspace: beam_moe_workspace_size(cfg, T,
 * BEAM_WEIGHTS_FP8). */
beam_status_t beam_moe_forward_fp8(const beam_moe_config_t *cfg, const void *hidden,
                                   const float *router_w, const float *corr_bias,
                                   const beam_fp8_weight_t *gate, const beam_fp8_weight_t *up,
                                   const beam_fp8_weight_t *down, void *out, int64_t T,
                                   void *workspace, size_t ws_bytes, void *stream);

/* MXFP8 expert weights of one projection (OCP MX format with E4M3
 * elements; the pages list MXFP8 beside FP8 as a precision Beam runs in:
 * "vLLM 实现 Reflection Beam 501B MoE 模型 Day 0 支持", the SkyRL paragraphs).
 * A weight is code x 2^(scale - 127), one E8M0 scale per 32 consecutive
 * elements along K. */
typedef struct {
  const uint8_t *q;     /* E4M3 codes [E, N, K]                                */
  const uint8_t *sf;    /* E8M0 scales of the [E*N, K/32] row-major matrix, in the
                           blocked order beam_moe_nvfp4_pack_scales writes for
                           S = K/32 (the same 128-row x 4-scale blocks)      */
} beam_mxfp8_weight_t;

/* The whole layer with MXFP8 experts.  Router and selection as in
 * beam_moe_forward; both expert GEMM inputs are quantised to MX blocks of 32
 * (x along d from its BF16 values before the gate/up GEMM, the FP32 SwiGLU
 * product along d_ff before the down GEMM) with the OCP MX conversion:
 * shared exponent X = floor(log2(amax)) - 8 clamped to [-127, 127] (-127 for
 * an all-zero block), codes E4M3(value * 2^-X), round to nearest even,
 * saturating at 448.  The GEMMs run as block-scaled E4M3 MMAs (one E8M0
 * scale per 32) with FP32 accumulation; the rest (FP32 routing weights, FP32
 * combine in slot order, one BF16 rounding) is beam_moe_forward's.  Extra
 * shape rule: d % 256 == 0.  Workspace: beam_moe_workspace_size(cfg, T,
 * BEAM_WEIGHTS_MXFP8). */
beam_status_t beam_moe_forward_mxfp8(const beam_moe_config_t *cfg, const void *hidden,
                                     const float *router_w, const float *corr_bias,
                                     const beam_mxfp8_weight_t *gate,
                                     const beam_mxfp8_weight_t *up,
                                     const beam_mxfp8_weight_t *down, void *out, int64_t T,
                                     void *workspace, size_t ws_bytes, void *stream);

/* The FP8 path's activation rule on its own: BF16 rows x [n, cols] ->
 * E4M3 codes q [n, cols] and FP32 scales [n] (cols % 8 == 0; all pointers
 * 16-byte aligned device memory).  n == 0 launches nothing. */
beam_status_t beam_moe_fp8_quantize_rows(const void *x, int64_t n, int32_t cols, uint8_t *q,
                                         float *scale, void *stream);

/* The quantised-expert layers followed by the decoder's sublayer boundary,
 * as beam_moe_forward_boundary is beam_moe_forward followed by it: the
 * boundary runs in the combine kernel on the layer's FP32 expert rows,
 * whatever format produced them, with the same arithmetic and the same
 * argument rules (boundary == NULL is the plain layer call).  The SGLang
 * post extends the fused norm / scaled-residual boundary to NVFP4 layers
 * (section "Fusion Optimizations", the kernel-fusion item).  Workspace and
 * weight rules as for the layer call of the same format. */
beam_status_t beam_moe_forward_nvfp4_boundary(const beam_moe_config_t *cfg, const void *hidden,
                                              const float *router_w, const float *corr_bias,
                                              const beam_fp4_weight_t *gate,
                                              const beam_fp4_weight_t *up,
                                              const beam_fp4_weight_t *down, void *out, int64_t T,
                                              const beam_moe_boundary_t *boundary,
                                              void *workspace, size_t ws_bytes, void *stream);
beam_status_t beam_moe_forward_nvfp4_a16_boundary(const beam_moe_config_t *cfg,
                                                  const void *hidden, const float *router_w,
                                                  const float *corr_bias,
                                                  const beam_fp4_weight_t *gate,
                                                  const beam_fp4_weight_t *up,
                                                  const beam_fp4_weight_t *down, void *out,
                                                  int64_t T, const beam_moe_boundary_t *boundary,
                                                  void *workspace, size_t ws_bytes, void *stream);
beam_status_t beam_moe_forward_fp8_boundary(const beam_moe_config_t *cfg, const void *hidden,
                                            const float *router_w, const float *corr_bias,
                                            const beam_fp8_weight_t *gate,
                                            const beam_fp8_weight_t *up,
                                            const beam_fp8_weight_t *down, void *out, int64_t T,
                                            const beam_moe_boundary_t *boundary, void *workspace,
                                            size_t ws_bytes, void *stream);
beam_status_t beam_moe_forward_mxfp8_boundary(const beam_moe_config_t *cfg, const void *hidden,
                                              const float *router_w, const float *corr_bias,
                                              const beam_mxfp8_weight_t *gate,
                                              const beam_mxfp8_weight_t *up,
                                              const beam_mxfp8_weight_t *down, void *out,
                                              int64_t T, const beam_moe_boundary_t *boundary,
                                              void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------- expert parallelism
 * Expert parallelism over n_ranks ranks ("SGLang 原生支持 Reflection 的 Beam
 * 并驱动其生产 API", section "Fusion Optimizations", the MegaMoE item and the
 * token-ownership figure after it: the experts are partitioned over the
 * ranks, a token's rows travel to the ranks that own its experts with
 * explicit expert ids and routing weights, every rank takes part even
 * without local tokens, and the complete outputs return to the token's
 * owning rank).  Rank q owns experts [q*E/n_ranks, (q+1)*E/n_ranks)
 * (n_ranks divides E).  One forward on n_ranks ranks is:
 *   1. beam_moe_ep_dispatch on every rank for its own tokens;
 *   2. an all-to-all of the packed rows, experts and weights (send_counts
 *      gives the split; the library performs no communication);
 *   3. beam_moe_ep_experts on every rank for the rows it received;
 *   4. the reverse all-to-all of the FP32 output rows, which come back in
 *      the order they were sent;
 *   5. beam_moe_ep_combine on every rank.
 * The result equals beam_moe_forward on the same tokens: the same
 * per-row arithmetic, the same slot-order FP32 sum and one BF16 rounding. */

/* Steps 1-2 of the layer on the tokens' owner, then the packing: one row per
 * (token, slot) pair, ordered by (expert, token, slot), which groups the rows
 * by owning rank.
 *   send_x      [T*topk, d] BF16  the pair's hidden row
 *   send_expert [T*topk]    int32 the pair's (global) expert
 *   send_w      [T*topk]    FP32  the pair's routing weight (alpha included)
 *   send_counts [n_ranks]   int32 rows bound for each rank, in rank order
 * All device buffers, caller-owned, 16-byte aligned.  The workspace is the
 * one beam_moe_workspace_size(cfg, T, BEAM_WEIGHTS_BF16) sizes; it must be
 * passed unchanged to beam_moe_ep_combine for the same T.  T == 0 writes
 * zero counts.  Asynchronous on `stream`. */
beam_status_t beam_moe_ep_dispatch(const beam_moe_config_t *cfg, const void *hidden,
                                   const float *router_w, const float *corr_bias, int64_t T,
                                   int32_t n_ranks, void *send_x, int32_t *send_expert,
                                   float *send_w, int32_t *send_counts, void *workspace,
                                   size_t ws_bytes, void *stream);

/* Workspace bytes of beam_moe_ep_experts (weight_fmt BEAM_WEIGHTS_BF16),
 * beam_moe_ep_experts_nvfp4 (BEAM_WEIGHTS_NVFP4) or beam_moe_ep_experts_fp8
 * (BEAM_WEIGHTS_FP8) for up to M_max received rows; 0 for an invalid
 * configuration or format. */
size_t beam_moe_ep_workspace_size(const beam_moe_config_t *cfg, int32_t n_ranks, int64_t M_max,
                                  int32_t weight_fmt);

/* Steps 3-4 of the layer on rank `rank` for M received rows:
 *   y_recv[i] = w_recv[i] * down(h), h = bf16(silu(x W_g^T) * (x W_u^T)),
 * with the expert expert_recv[i], x = x_recv[i] (BF16 [M, d]), in FP32
 * ([M, d], row i for received row i).  w_gate / w_up [E/n_ranks, d_ff, d]
 * and w_down [E/n_ranks, d, d_ff] hold this rank's experts only.  An
 * expert id outside the rank's range latches BEAM_ERR_DEVICE_CHECK and its
 * row is not written.  M == 0 launches nothing. */
beam_status_t beam_moe_ep_experts(const beam_moe_config_t *cfg, int32_t n_ranks, int32_t rank,
                                  const void *x_recv, const int32_t *expert_recv,
                                  const float *w_recv, const void *w_gate, const void *w_up,
                                  const void *w_down, float *y_recv, int64_t M, void *workspace,
                                  size_t ws_bytes, void *stream);

/* beam_moe_ep_experts with NVFP4 expert weights (the pages' MegaMoE path
 * runs Beam's NVFP4 experts): the rank's received rows are quantised to
 * NVFP4 and go through the block-scaled FP4 GEMMs of beam_moe_forward_nvfp4;
 * gate / up / down describe this rank's E/n_ranks experts (codes
 * [E/n_ranks, N, K/2], their blocked scales, global scales [E/n_ranks]).
 * Extra shape rules: d % 256 == 0, d_ff % 256 == 0. */
beam_status_t beam_moe_ep_experts_nvfp4(const beam_moe_config_t *cfg, int32_t n_ranks,
                                        int32_t rank, const void *x_recv,
                                        const int32_t *expert_recv, const float *w_recv,
                                        const beam_fp4_weight_t *gate, const beam_fp4_weight_t *up,
                                        const beam_fp4_weight_t *down, float *y_recv, int64_t M,
                                        void *workspace, size_t ws_bytes, void *stream);

/* beam_moe_ep_experts with dynamic FP8 expert weights (beyond the pages,
 * whose expert-parallel MegaMoE path leaves dynamic FP8 out): each received
 * row is quantised to E4M3 with its own scale (a row per token and slot, so
 * the token's codes and scale) and goes through the FP8 GEMMs of
 * beam_moe_forward_fp8; gate / up / down describe this rank's E/n_ranks
 * experts (codes [E/n_ranks, N, K], row scales [E/n_ranks, N]). */
beam_status_t beam_moe_ep_experts_fp8(const beam_moe_config_t *cfg, int32_t n_ranks,
                                      int32_t rank, const void *x_recv,
                                      const int32_t *expert_recv, const float *w_recv,
                                      const beam_fp8_weight_t *gate, const beam_fp8_weight_t *up,
                                      const beam_fp8_weight_t *down, float *y_recv, int64_t M,
                                      void *workspace, size_t ws_bytes, void *stream);

/* The owner's combine: out[t] = bf16(sum over slots, in slot order, of the
 * returned FP32 rows), y_back [T*topk, d] in the order beam_moe_ep_dispatch
 * packed them.  `workspace` is the dispatch call's, unchanged. */
beam_status_t beam_moe_ep_combine(const beam_moe_config_t *cfg, const float *y_back, int64_t T,
                                  void *out, void *workspace, size_t ws_bytes, void *stream);

/* Synchronises `stream`, returns the workspace's latched status and clears
 * it.  The only entry point that waits for the device. */
beam_status_t beam_moe_check_status(void *workspace, void *stream);

/* Profiling aid: when n >= 8 events (cudaEvent_t) are given, every later
 * beam_moe_forward / beam_moe_forward_routed records them on its stream at
 * the step boundaries: [0] start, [1] router, [2] selection, [3] permute,
 * [4] token rows (BF16: their scatter into expert order when T*topk > 4*E,
 * smaller batches gather inside the gate/up GEMM; NVFP4 and FP8: their
 * quantisation, then for FP8 the scatter), [5] gate/up GEMM, [6] down GEMM,
 * [7] combine (each after its step).  Steps a call does not run record at the same point as the previous
 * one.  Below 256 tokens (at most 256 experts) the router, the selection and
 * the permutation are one cooperative launch: [1], [2] and [3] are all
 * recorded after it.  While `stream` is being captured into a CUDA graph
 * the records become event-record nodes (cudaEventRecordExternal), so each
 * replay timestamps them again.  n == 0 switches it off.  Process-wide; not
 * thread-safe. */
beam_status_t beam_moe_set_stage_events(void *const *events, int32_t n);

/* Test aid for the bounded waits: wait_limit_us bounds every device-side
 * wait of the expert GEMMs (0 restores the default of two seconds);
 * withhold_first_load != 0 makes the first CTA of the next gate/up GEMM skip
 * its first operand load, so its MMA wait runs out and the call latches
 * BEAM_ERR_TIMEOUT without faulting.  Process-wide; not thread-safe. */
beam_status_t beam_moe_set_debug(uint32_t wait_limit_us, int32_t withhold_first_load);

/* Number of kernels one call of T tokens launches (for accounting):
 * beam_moe_forward (and beam_moe_forward_noalloc) for weight_fmt
 * BEAM_WEIGHTS_BF16, beam_moe_forward_nvfp4 for BEAM_WEIGHTS_NVFP4,
 * beam_moe_forward_nvfp4_a16 for BEAM_WEIGHTS_NVFP4_A16,
 * beam_moe_forward_fp8 for BEAM_WEIGHTS_FP8, beam_moe_forward_mxfp8 for
 * BEAM_WEIGHTS_MXFP8, and with
 * routed != 0 beam_moe_forward_routed (BF16 only).  Returns 0 for an invalid
 * configuration, T <= 0 or an unknown combination.  Host-only. */
int32_t beam_moe_kernels_per_forward(const beam_moe_config_t *cfg, int64_t T, int32_t weight_fmt,
                                     int32_t routed);

const char *beam_status_string(beam_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* BEAM_MOE_H_ */
