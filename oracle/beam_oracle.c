/*
 * Beam MoE layer: plain CPU oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * This is the slow, obviously correct reference the CUDA path is checked
 * against.  Only the tests, the package smoke check and the benchmark's CPU
 * baseline load it; the product path never does.  It shares no code, header,
 * table or constant generator with the CUDA library.
 *
 * Sources (page title, section):
 *   [SGL]  "SGLang 原生支持 Reflection 的 Beam 并驱动其生产 API",
 *          sections "Dense Layers and Grouped MoE Routing",
 *          "BF16 MoE Kernel Optimization", "Fusion Optimizations",
 *          "Sandwich Normalization and Depth-Scaled Residuals".
 *   [VLLM] "vLLM 实现 Reflection Beam 501B MoE 模型 Day 0 支持",
 *          sections "MoE and residual stream", "Agent-driven optimization".
 *   [HF]   "Reflection 发布 501B 开源模型 Beam，Apache 2.0 许可",
 *          sections "专家混合" (mixture of experts) and "残差流" (residual
 *          stream: router and SwiGLU product computed in FP32).
 *   [HWC]  "Reflection Beam 技术笔记：501B MoE 如何把「大容量」和「可部署」拧在一起",
 *          section 1 (sparse MoE).
 *
 * Precision convention: every dot product accumulates in double and is
 * rounded once to the precision the pages fix (FP32 router logits, FP32
 * gate/up accumulators, FP32 SwiGLU product, BF16 activation h, FP32 routing
 * weights, BF16 layer output).  Where the pages leave a step open the reading
 * taken is stated at the function.  Built with -ffp-contract=off so that no
 * multiply-add is fused and x86-64 and aarch64 give identical bits.
 *
 * Parity status: every function here is pinned by the CPU test-suite
 * (library routines, brute force, closed forms, invariants); none is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                            */
/* ------------------------------------------------------------------------ */

/* BF16 is the top half of an IEEE binary32. */
static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a binary32 to the nearest BF16, ties to even (NaN stays NaN). */
static uint16_t bf16_round(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t keep = u >> 16;
  uint32_t rest = u & 0xffffu;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

/* Nearest BF16 of a double, ties to even, with one rounding: the double is
 * first brought to binary32 by rounding to odd (truncate, then set the last
 * bit when inexact), which keeps the later rounding to 8 bits correct. */
static uint16_t bf16_round_double(double v) {
  float f = (float)v;
  if ((double)f != v) {
    if (fabs((double)f) > fabs(v)) f = nextafterf(f, 0.0f);
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u |= 1u;
    memcpy(&f, &u, sizeof f);
  }
  return bf16_round(f);
}

/* Nearest IEEE binary16 value of a double, ties to even, with subnormals;
 * magnitudes beyond the largest finite binary16 (65504) saturate to it.
 * Written from the format: 11 significant bits, exponents -14..15, spacing
 * 2^-24 below 2^-14. */
static double f16_round_value(double v) {
  if (v != v) return v;
  const double a = fabs(v);
  if (a >= 65504.0) return v < 0 ? -65504.0 : 65504.0;
  if (a == 0.0) return v;
  int e;
  frexp(a, &e);                      /* a in [2^(e-1), 2^e) */
  int q = e - 1 - 10;                /* spacing exponent for 11 significant bits */
  if (q < -24) q = -24;              /* subnormal spacing */
  const double step = ldexp(1.0, q);
  double n = floor(a / step);        /* exact: a / step is a scaling by a power of two */
  const double rest = a - n * step;
  if (rest > step / 2 || (rest == step / 2 && fmod(n, 2.0) != 0.0)) n += 1.0;
  double r = n * step;
  if (r > 65504.0) r = 65504.0;
  return v < 0 ? -r : r;
}

/* E2M1 (FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * Magnitudes of codes 0..7 written out from the format definition. */
static double e2m1_value(uint8_t code) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double m = mag[code & 7u];
  return (code & 8u) ? -m : m;
}

/* E4M3 (FP8, "fn" flavour): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, largest finite 448. */
static double e4m3_value(uint8_t code) {
  int sign = (code >> 7) & 1;
  int ex = (code >> 3) & 15;
  int man = code & 7;
  double v;
  if (ex == 15 && man == 7) return NAN;
  if (ex == 0)
    v = ldexp((double)man / 8.0, -6);
  else
    v = ldexp(1.0 + (double)man / 8.0, ex - 7);
  return sign ? -v : v;
}

/* E8M0 (the shared scale of the MX formats): 8 exponent bits, bias 127, no
 * sign and no mantissa; code 255 is NaN. */
static double e8m0_value(uint8_t code) {
  if (code == 0xFFu) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* Nearest code by exhaustive search over the format's finite magnitudes,
 * ties to the even code (the one whose lowest bit is 0); values beyond the
 * largest finite magnitude saturate to it (satfinite).  Brute force on
 * purpose: it is the definition of round-to-nearest-even. */
static uint8_t nearest_code(double a, double (*val)(uint8_t), int n_finite) {
  int best = 0;
  double best_err = fabs(a - val(0));
  for (int c = 1; c < n_finite; ++c) {
    double err = fabs(a - val((uint8_t)c));
    if (err < best_err || (err == best_err && (best & 1) && !(c & 1))) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)best;
}

static uint8_t e2m1_encode(float v) {
  if (isnan(v)) return 0;
  if (isinf(v)) return (uint8_t)(v < 0 ? 15u : 7u);
  uint8_t c = nearest_code(fabs((double)v), e2m1_value, 8);
  return (uint8_t)(signbit(v) ? (c | 8u) : c);
}

static uint8_t e4m3_encode(float v) {
  if (isnan(v)) return 0x7f;
  if (isinf(v)) return (uint8_t)(v < 0 ? 0xfeu : 0x7eu);
  uint8_t c = nearest_code(fabs((double)v), e4m3_value, 127);
  return (uint8_t)(signbit(v) ? (c | 0x80u) : c);
}

/* ------------------------------------------------------------------------ */
/* Router: [SGL] "The router computes FP32 logits"; [VLLM] "FP32 router.  The */
/* 5120 x 256 router weights, accumulation, and logits are all FP32".        */
/* logits[t,e] = sum_j x[t,j] * W_r[e,j], accumulated in double, rounded     */
/* once to FP32.  W_r is stored [E, d] (nn.Linear layout).                   */
/* ------------------------------------------------------------------------ */
int oracle_router_logits(const uint16_t *x, const float *wr, int64_t T,
                         int32_t d, int32_t E, float *logits) {
  if (T < 0 || d <= 0 || E <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    const uint16_t *xr = x + t * (int64_t)d;
    for (int32_t e = 0; e < E; ++e) {
      const float *wrow = wr + (int64_t)e * d;
      double acc = 0.0;
      for (int32_t j = 0; j < d; ++j) acc += bf16_value(xr[j]) * (double)wrow[j];
      logits[t * (int64_t)E + e] = (float)acc;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Group-limited selection.                                                  */
/*   [SGL] grouped top-k uses sigmoid scores and an expert correction bias   */
/*         to choose the experts; FP32 routing coefficients; the routed      */
/*         scale is applied at combine or carried in the weights.            */
/*   [VLLM] sigmoid scores plus a correction bias pick the best 4 of 8       */
/*         groups, then the top 8 experts; renormalised weights x 2.5; no    */
/*         shared expert.                                                    */
/*   [HF]  groups ranked by the sum of each group's top two scores.          */
/* Readings where the pages are silent:                                      */
/*   - the group score and the expert choice use c = s + b (one FP32 add);  */
/*   - the combine weights use s, not c (the bias only chooses);             */
/*   - ties: the order is total on (value descending, index ascending);      */
/*   - the scale 2.5 is carried in the FP32 weights;                         */
/*   - slot order of the chosen experts is that same (c desc, e asc) order.  */
/* Per token it also reports the two margins parity tests exempt on:         */
/*   expert_margin = c(k-th chosen) - c(best unchosen candidate in the kept  */
/*   groups), group_margin = gs(kg-th kept) - gs(best dropped group); +inf   */
/*   when nothing is left to compare with.                                   */
/* ------------------------------------------------------------------------ */
static int ranks_before(float va, int32_t ia, float vb, int32_t ib) {
  return va > vb || (va == vb && ia < ib);
}

int oracle_route(const float *logits, const float *bias, int64_t T, int32_t E,
                 int32_t G, int32_t kg, int32_t k, float alpha, int32_t *idx,
                 float *w, float *s_out, float *c_out, uint8_t *keep_out,
                 double *expert_margin, double *group_margin) {
  if (T < 0 || E <= 0 || G <= 0 || E % G != 0) return -1;
  const int32_t S = E / G;
  if (S < 2 || kg < 1 || kg > G || k < 1 || k > kg * S) return -1;
  int err = 0;
#pragma omp parallel
  {
    float *s = (float *)malloc(sizeof(float) * (size_t)E);
    float *c = (float *)malloc(sizeof(float) * (size_t)E);
    float *gs = (float *)malloc(sizeof(float) * (size_t)G);
    uint8_t *keep = (uint8_t *)malloc((size_t)G);
    uint8_t *taken = (uint8_t *)malloc((size_t)E);
    if (!s || !c || !gs || !keep || !taken) {
#pragma omp atomic write
      err = -3;
    } else {
#pragma omp for schedule(static)
      for (int64_t t = 0; t < T; ++t) {
        const float *lg = logits + t * (int64_t)E;
        /* scores and choice scores */
        for (int32_t e = 0; e < E; ++e) {
          s[e] = (float)(1.0 / (1.0 + exp(-(double)lg[e])));
          c[e] = s[e] + bias[e];
        }
        /* group score = top-1 + top-2 choice score inside the group */
        for (int32_t g = 0; g < G; ++g) {
          int32_t b1 = -1, b2 = -1;
          for (int32_t e = g * S; e < (g + 1) * S; ++e) {
            if (b1 < 0 || ranks_before(c[e], e, c[b1], b1)) {
              b2 = b1;
              b1 = e;
            } else if (b2 < 0 || ranks_before(c[e], e, c[b2], b2)) {
              b2 = e;
            }
          }
          gs[g] = c[b1] + c[b2];
        }
        /* keep the best kg groups */
        memset(keep, 0, (size_t)G);
        int32_t last_kept = -1;
        for (int32_t r = 0; r < kg; ++r) {
          int32_t best = -1;
          for (int32_t g = 0; g < G; ++g)
            if (!keep[g] && (best < 0 || ranks_before(gs[g], g, gs[best], best))) best = g;
          keep[best] = 1;
          last_kept = best;
        }
        {
          int32_t next = -1;
          for (int32_t g = 0; g < G; ++g)
            if (!keep[g] && (next < 0 || ranks_before(gs[g], g, gs[next], next))) next = g;
          group_margin[t] = next < 0 ? INFINITY : (double)gs[last_kept] - (double)gs[next];
        }
        /* top-k experts among the kept groups' members */
        memset(taken, 0, (size_t)E);
        double ssum = 0.0;
        int32_t *ti = idx + t * (int64_t)k;
        for (int32_t r = 0; r < k; ++r) {
          int32_t best = -1;
          for (int32_t e = 0; e < E; ++e)
            if (keep[e / S] && !taken[e] && (best < 0 || ranks_before(c[e], e, c[best], best)))
              best = e;
          taken[best] = 1;
          ti[r] = best;
          ssum += (double)s[best];
        }
        {
          int32_t next = -1;
          for (int32_t e = 0; e < E; ++e)
            if (keep[e / S] && !taken[e] && (next < 0 || ranks_before(c[e], e, c[next], next)))
              next = e;
          expert_margin[t] = next < 0 ? INFINITY : (double)c[ti[k - 1]] - (double)c[next];
        }
        /* renormalised weights over s, times the routed scale */
        for (int32_t r = 0; r < k; ++r)
          w[t * (int64_t)k + r] = (float)((double)alpha * (double)s[ti[r]] / ssum);
        if (s_out) memcpy(s_out + t * (int64_t)E, s, sizeof(float) * (size_t)E);
        if (c_out) memcpy(c_out + t * (int64_t)E, c, sizeof(float) * (size_t)E);
        if (keep_out) memcpy(keep_out + t * (int64_t)G, keep, (size_t)G);
      }
    }
    free(s);
    free(c);
    free(gs);
    free(keep);
    free(taken);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Experts and combine.                                                      */
/*   [HF] each expert is a SwiGLU MLP of intermediate size 2560; the         */
/*        SwiGLU product is computed in FP32; outputs are combined with the  */
/*        normalised router weights times 2.5 ([VLLM]: no shared expert).    */
/*   [SGL] "BF16 MoE Kernel Optimization": gate/up and activation keep BF16  */
/*        rounding boundaries; FP32 routing weights are applied before the   */
/*        down output is rounded; [SGL] "Fusion Optimizations": local expert */
/*        summation, routed scaling and BF16 rounding.                       */
/* Readings: SwiGLU(x) = silu(x W_g^T) * (x W_u^T), silu(z) = z/(1+e^-z);    */
/* g and u are the FP32-rounded accumulators (not rounded to BF16); the      */
/* product is rounded to FP32 and then to BF16 (h, the down GEMM's input);   */
/* the down accumulation, the weighting and the sum over the k slots stay in */
/* double; the output is that double sum rounded once to BF16.               */
/* Weight layouts (nn.Linear): W_g, W_u [F, d] and W_d [d, F] per expert,    */
/* passed as one pointer per expert (NULL for experts nobody uses).          */
/* tokens: optional list of rows to compute (NULL = all T rows); rows not    */
/* listed are left untouched in out.  out_exact (optional, [T, d] double)    */
/* receives the output before its final rounding.                            */
/* ------------------------------------------------------------------------ */
typedef struct {
  /* BF16 weights */
  const uint16_t *const *wg, *const *wu, *const *wd;
  /* NVFP4 weights: packed E2M1 codes (low nibble = even column), one E4M3
   * scale per 16 consecutive elements along K, one FP32 global scale per
   * expert and projection. */
  const uint8_t *const *qg, *const *qu, *const *qd;
  const uint8_t *const *sfg, *const *sfu, *const *sfd;
  const float *gsg, *gsu, *gsd;
  /* FP8 weights: E4M3 codes [N, K], one FP32 scale per output row [N]. */
  const uint8_t *const *eg, *const *eu, *const *ed;
  const float *const *seg, *const *seu, *const *sed;
  /* MXFP8 weights: E4M3 codes [N, K], one E8M0 scale per 32 consecutive
   * elements along K [N, K/32]. */
  const uint8_t *const *mg, *const *mu, *const *md;
  const uint8_t *const *smg, *const *smu, *const *smd;
  int fp4;
  int fp8;
  int mx;
  int act_quant;
  /* FP8 near ties (optional): per token the summed effect on each output of
   * the h codes that a rounding of h on the other side of a BF16 midpoint
   * would move, and a flag for rows whose scale could move. */
  double tie_rel;
  double *tie_slack;   /* [T, d] */
  uint8_t *scale_tie;  /* [T] */
} weights_t;

/* One row of the dynamic FP8 scheme's activation rule (per token, or per
 * (token, expert) row of the down GEMM's input): scale = amax / 448 in FP32
 * (1 for an all-zero row), code_i = E4M3(v_i / scale) with FP32 divisions,
 * round to nearest even, saturating at 448.  The E4M3 magnitudes are tabled
 * from the format definition once per row; the search over them is the same
 * exhaustive nearest-even rule as e4m3_encode.  Writes codes and scale when
 * asked, and the dequantised values code * scale when out is given. */
static void fp8_row_quantize(const float *v, int64_t n, uint8_t *q, float *scale_out,
                             double *out) {
  double mag[127];
  for (int c = 0; c < 127; ++c) mag[c] = e4m3_value((uint8_t)c);
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int64_t i = 0; i < n; ++i) {
    const float r = v[i] / scale;
    const double a = fabs((double)r);
    int best = 0;
    double best_err = fabs(a - mag[0]);
    for (int c = 1; c < 127; ++c) {
      double err = fabs(a - mag[c]);
      if (err < best_err || (err == best_err && (best & 1) && !(c & 1))) {
        best = c;
        best_err = err;
      }
    }
    const uint8_t code = (uint8_t)(signbit(r) ? (best | 0x80) : best);
    if (q) q[i] = code;
    if (out) out[i] = e4m3_value(code) * (double)scale;
  }
  if (scale_out) *scale_out = scale;
}

/* The values of all 256 E4M3 and all 16 E2M1 codes, tabled from the
 * decoders above (the weight loops look codes up here instead of decoding
 * each one again).  Filled by experts_impl before its parallel region. */
static double e4m3_tab[256];
static double e2m1_tab[16];

static void fill_format_tables(void) {
  for (int c = 0; c < 256; ++c) e4m3_tab[c] = e4m3_value((uint8_t)c);
  for (int c = 0; c < 16; ++c) e2m1_tab[c] = e2m1_value((uint8_t)c);
}

static double fp8_weight(const uint8_t *q, const float *s, int64_t row, int64_t col, int64_t K) {
  return e4m3_tab[q[row * K + col]] * (double)s[row];
}

/* Near ties of the FP8 path's h quantisation.  hf holds one (token, expert)
 * row of FP32 SwiGLU products and hb their BF16 roundings.  An element whose
 * FP32 value lies within rel * |value| of the midpoint between its BF16
 * value and the next BF16 value on its side could be rounded to that
 * neighbour by an FP32 computation whose error is below that bound.  For
 * such an element diff receives the change of its dequantised E4M3 value if
 * the neighbour were taken (0 when both quantise alike); when the neighbour
 * or the element itself decides the row's amax, the row's scale could move
 * and *scale_flag is set instead. */
static void fp8_h_ties(const float *hf, const float *hb, int64_t n, double rel, double *diff,
                       int *scale_flag) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(hb[i]);
    if (a > amax) amax = a;
  }
  const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int64_t i = 0; i < n; ++i) {
    diff[i] = 0.0;
    const double v = (double)hf[i], b = (double)hb[i];
    if (v == b || v != v) continue;
    const uint16_t mag = (uint16_t)(bf16_round(hf[i]) & 0x7fffu);
    const uint16_t nmag = fabs(v) > fabs(b) ? (uint16_t)(mag + 1u) : (uint16_t)(mag - 1u);
    const double nb = bf16_value((uint16_t)((v < 0 ? 0x8000u : 0u) | nmag));
    if (fabs(v - 0.5 * (b + nb)) > rel * fabs(v)) continue;
    if (fabs(nb) >= (double)amax || fabs(b) == (double)amax) {
      *scale_flag = 1;
      continue;
    }
    const double qb = e4m3_value(e4m3_encode((float)b / scale)) * (double)scale;
    const double qn = e4m3_value(e4m3_encode((float)nb / scale)) * (double)scale;
    diff[i] = qn - qb;
  }
}

/* One MX block ([OCP] "Microscaling Formats (MX) v1.0", the conversion of a
 * vector of scalars to an MX block), E4M3 elements: the shared exponent is
 * X = floor(log2(amax)) - 8 (8 = the largest exponent of E4M3), clamped to
 * the E8M0 range [-127, 127] (an all-zero block takes -127); each element is
 * E4M3(v / 2^X), nearest even, saturating at 448.  Writes the scale code, the
 * element codes (when asked) and the dequantised values code * 2^X. */
static int mx_shared_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  int e;
  frexp((double)amax, &e);             /* amax in [2^(e-1), 2^e) */
  int x = e - 1 - 8;
  return x < -127 ? -127 : x > 127 ? 127 : x;
}

static void mx_block_quantize(const float *v, int n, uint8_t *scale_code, uint8_t *codes,
                              double *out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  const int x = mx_shared_exponent(amax);
  if (scale_code) *scale_code = (uint8_t)(x + 127);
  for (int i = 0; i < n; ++i) {
    const float r = (float)ldexp((double)v[i], -x);   /* exact: a power-of-two scaling */
    const uint8_t c = e4m3_encode(r);
    if (codes) codes[i] = c;
    if (out) out[i] = e4m3_value(c) * ldexp(1.0, x);
  }
}

/* Near ties of the MXFP8 path's h quantisation (see fp8_h_ties for the
 * FP8 path): an FP32 h element whose scaled value lies within rel of an E4M3
 * rounding midpoint gets in diff the change of its dequantised value if the
 * neighbouring code were taken; a block whose amax lies within rel of a
 * power of two (where the shared exponent changes) sets *scale_flag. */
static void mx_h_ties(const float *hf, int n, double rel, double *diff, int *scale_flag) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(hf[i]);
    if (a > amax) amax = a;
  }
  if (amax > 0.0f) {
    int e;
    const double m = frexp((double)amax, &e);       /* amax = m 2^e, m in [0.5, 1) */
    if (m - 0.5 <= rel * m || 1.0 - m <= rel * m) *scale_flag = 1;
  }
  const int x = mx_shared_exponent(amax);
  for (int i = 0; i < n; ++i) {
    diff[i] = 0.0;
    const double r = fabs(ldexp((double)hf[i], -x));
    if (r == 0.0 || r >= 448.0) continue;
    const int c = e4m3_encode((float)r) & 0x7f;
    const double vc = e4m3_value((uint8_t)c);
    if (r == vc) continue;
    const int nb = r > vc ? c + 1 : c - 1;
    if (nb < 0 || nb > 126) continue;
    const double vn = e4m3_value((uint8_t)nb);
    if (fabs(r - 0.5 * (vc + vn)) > rel * r) continue;
    diff[i] = (hf[i] < 0 ? -1.0 : 1.0) * (vn - vc) * ldexp(1.0, x);
  }
}

static double mx_weight(const uint8_t *q, const uint8_t *sc, int64_t row, int64_t col, int64_t K) {
  return e4m3_tab[q[row * K + col]] * ldexp(1.0, (int)sc[row * (K / 32) + col / 32] - 127);
}

/* One NVFP4 block of 16: the activation rule used on both GEMM inputs of the
 * NVFP4 path (global scale 1): scale = E4M3(amax / 6), code_i =
 * E2M1(v_i / scale) with FP32 divisions, all-zero codes when the scale
 * rounds to 0.  Writes the dequantised values. */
static void nvfp4_block_roundtrip(const float *v, double *out16) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  uint8_t sf = e4m3_encode(amax / 6.0f);
  float scale = (float)e4m3_value(sf);
  for (int i = 0; i < 16; ++i) {
    uint8_t q = scale > 0.0f ? e2m1_encode(v[i] / scale) : 0;
    out16[i] = e2m1_value(q) * (double)scale;
  }
}

static double fp4_weight(const uint8_t *q, const uint8_t *sf, float gs,
                         int64_t row, int64_t col, int64_t K) {
  int64_t flat = row * K + col;
  uint8_t byte = q[flat >> 1];
  uint8_t code = (flat & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15u);
  return e2m1_tab[code] * e4m3_tab[sf[row * (K / 16) + col / 16]] * (double)gs;
}

static int experts_impl(const uint16_t *x, int64_t T, int32_t d, int32_t F,
                        int32_t k, int32_t E, const int32_t *idx, const float *w,
                        const weights_t *W, const int64_t *tokens,
                        int64_t n_tokens, uint16_t *out, double *out_exact) {
  if (T < 0 || d <= 0 || F <= 0 || k <= 0 || (d % 16) || (F % 16)) return -1;
  if (W->mx && ((d % 32) || (F % 32))) return -1;
  const int64_t n = tokens ? n_tokens : T;
  int err = 0;
  /* every referenced expert must have its weights */
  for (int64_t i = 0; i < n && !err; ++i) {
    int64_t t = tokens ? tokens[i] : i;
    if (t < 0 || t >= T) { err = -1; break; }
    for (int32_t j = 0; j < k; ++j) {
      int32_t e = idx[t * k + j];
      if (e < 0 || e >= E) { err = -1; break; }
      if (W->fp4   ? (!W->qg[e] || !W->qu[e] || !W->qd[e])
          : W->fp8 ? (!W->eg[e] || !W->eu[e] || !W->ed[e])
          : W->mx  ? (!W->mg[e] || !W->mu[e] || !W->md[e])
                   : (!W->wg[e] || !W->wu[e] || !W->wd[e])) {
        err = -2;
        break;
      }
    }
  }
  if (err) return err;
  fill_format_tables();
#pragma omp parallel
  {
    double *xin = (double *)malloc(sizeof(double) * (size_t)d);
    float *hf = (float *)malloc(sizeof(float) * (size_t)F);
    double *hin = (double *)malloc(sizeof(double) * (size_t)F);
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    float *tmp = (float *)malloc(sizeof(float) * (size_t)(d > F ? d : F));
    double *hdiff = W->tie_slack ? (double *)malloc(sizeof(double) * (size_t)F) : NULL;
    double *slack = W->tie_slack ? (double *)malloc(sizeof(double) * (size_t)d) : NULL;
    int32_t *tie_f = W->tie_slack ? (int32_t *)malloc(sizeof(int32_t) * (size_t)F) : NULL;
    if (!xin || !hf || !hin || !acc || !tmp ||
        (W->tie_slack && (!hdiff || !slack || !tie_f))) {
#pragma omp atomic write
      err = -3;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        const uint16_t *xr = x + t * (int64_t)d;
        /* the expert input row (NVFP4 path may quantise it, or take it in
           F16 for the F16 tensor-core operands) */
        if (W->fp8 && W->act_quant) {
          for (int32_t j = 0; j < d; ++j) tmp[j] = (float)bf16_value(xr[j]);
          fp8_row_quantize(tmp, d, NULL, NULL, xin);
        } else if (W->fp4 && W->act_quant == 2) {
          for (int32_t j = 0; j < d; ++j) xin[j] = f16_round_value(bf16_value(xr[j]));
        } else if (W->fp4 && W->act_quant) {
          for (int32_t j = 0; j < d; ++j) tmp[j] = (float)bf16_value(xr[j]);
          for (int32_t j = 0; j < d; j += 16) nvfp4_block_roundtrip(tmp + j, xin + j);
        } else if (W->mx && W->act_quant) {
          for (int32_t j = 0; j < d; ++j) tmp[j] = (float)bf16_value(xr[j]);
          for (int32_t j = 0; j < d; j += 32) mx_block_quantize(tmp + j, 32, NULL, NULL, xin + j);
        } else {
          for (int32_t j = 0; j < d; ++j) xin[j] = bf16_value(xr[j]);
        }
        for (int32_t j = 0; j < d; ++j) acc[j] = 0.0;
        int scale_flag = 0;
        if (slack)
          for (int32_t j = 0; j < d; ++j) slack[j] = 0.0;
        for (int32_t slot = 0; slot < k; ++slot) {
          const int32_t e = idx[t * k + slot];
          const double wt = (double)w[t * k + slot];
          /* gate/up accumulators (FP32) and the SwiGLU product (FP32) */
          for (int32_t f = 0; f < F; ++f) {
            double ga = 0.0, ua = 0.0;
            if (W->fp4) {
              for (int32_t j = 0; j < d; ++j) {
                ga += xin[j] * fp4_weight(W->qg[e], W->sfg[e], W->gsg[e], f, j, d);
                ua += xin[j] * fp4_weight(W->qu[e], W->sfu[e], W->gsu[e], f, j, d);
              }
            } else if (W->fp8) {
              for (int32_t j = 0; j < d; ++j) {
                ga += xin[j] * fp8_weight(W->eg[e], W->seg[e], f, j, d);
                ua += xin[j] * fp8_weight(W->eu[e], W->seu[e], f, j, d);
              }
            } else if (W->mx) {
              for (int32_t j = 0; j < d; ++j) {
                ga += xin[j] * mx_weight(W->mg[e], W->smg[e], f, j, d);
                ua += xin[j] * mx_weight(W->mu[e], W->smu[e], f, j, d);
              }
            } else {
              const uint16_t *gr = W->wg[e] + (int64_t)f * d;
              const uint16_t *ur = W->wu[e] + (int64_t)f * d;
              for (int32_t j = 0; j < d; ++j) {
                ga += xin[j] * bf16_value(gr[j]);
                ua += xin[j] * bf16_value(ur[j]);
              }
            }
            const double g = (double)(float)ga;
            const double u = (double)(float)ua;
            const double silu = g / (1.0 + exp(-g));
            hf[f] = (float)(silu * u);
          }
          /* the down GEMM's input */
          if (W->fp8 && W->act_quant) {
            /* h keeps its BF16 rounding, then the row is quantised */
            for (int32_t f = 0; f < F; ++f) tmp[f] = (float)bf16_value(bf16_round(hf[f]));
            fp8_row_quantize(tmp, F, NULL, NULL, hin);
            if (slack) {
              int32_t n_tie = 0;
              fp8_h_ties(hf, tmp, F, W->tie_rel, hdiff, &scale_flag);
              for (int32_t f = 0; f < F; ++f)
                if (hdiff[f] != 0.0) tie_f[n_tie++] = f;
              /* each near tie's whole effect on every output of the token */
              for (int32_t q = 0; q < n_tie; ++q)
                for (int32_t r = 0; r < d; ++r)
                  slack[r] += fabs(wt * hdiff[tie_f[q]] * fp8_weight(W->ed[e], W->sed[e], r,
                                                                      tie_f[q], F));
            }
          } else if (W->mx && W->act_quant) {
            /* the FP32 product itself, per 32 along F */
            for (int32_t f = 0; f < F; f += 32) mx_block_quantize(hf + f, 32, NULL, NULL, hin + f);
            if (slack) {
              int32_t n_tie = 0;
              for (int32_t f = 0; f < F; f += 32)
                mx_h_ties(hf + f, 32, W->tie_rel, hdiff + f, &scale_flag);
              for (int32_t f = 0; f < F; ++f)
                if (hdiff[f] != 0.0) tie_f[n_tie++] = f;
              for (int32_t q = 0; q < n_tie; ++q)
                for (int32_t r = 0; r < d; ++r)
                  slack[r] += fabs(wt * hdiff[tie_f[q]] * mx_weight(W->md[e], W->smd[e], r,
                                                                     tie_f[q], F));
            }
          } else if (W->fp4 && W->act_quant == 2) {
            for (int32_t f = 0; f < F; ++f) hin[f] = f16_round_value((double)hf[f]);
          } else if (W->fp4 && W->act_quant) {
            for (int32_t f = 0; f < F; f += 16) nvfp4_block_roundtrip(hf + f, hin + f);
          } else {
            for (int32_t f = 0; f < F; ++f) hin[f] = bf16_value(bf16_round(hf[f]));
          }
          /* down projection, weighted, summed over the slots in double */
          for (int32_t r = 0; r < d; ++r) {
            double ya = 0.0;
            if (W->fp4) {
              for (int32_t f = 0; f < F; ++f)
                ya += hin[f] * fp4_weight(W->qd[e], W->sfd[e], W->gsd[e], r, f, F);
            } else if (W->fp8) {
              for (int32_t f = 0; f < F; ++f)
                ya += hin[f] * fp8_weight(W->ed[e], W->sed[e], r, f, F);
            } else if (W->mx) {
              for (int32_t f = 0; f < F; ++f)
                ya += hin[f] * mx_weight(W->md[e], W->smd[e], r, f, F);
            } else {
              const uint16_t *dr = W->wd[e] + (int64_t)r * F;
              for (int32_t f = 0; f < F; ++f) ya += hin[f] * bf16_value(dr[f]);
            }
            acc[r] += wt * ya;
          }
        }
        for (int32_t r = 0; r < d; ++r) out[t * (int64_t)d + r] = bf16_round_double(acc[r]);
        if (out_exact)
          for (int32_t r = 0; r < d; ++r) out_exact[t * (int64_t)d + r] = acc[r];
        if (slack) {
          for (int32_t r = 0; r < d; ++r) W->tie_slack[t * (int64_t)d + r] = slack[r];
          W->scale_tie[t] = (uint8_t)scale_flag;
        }
      }
    }
    free(xin);
    free(hf);
    free(hin);
    free(acc);
    free(tmp);
    free(hdiff);
    free(slack);
    free(tie_f);
  }
  return err;
}

/* The gate/up step of one expert on n rows alone, as the expert layer takes
 * it ([SGL] "BF16 MoE Kernel Optimization"; [HF] "残差流": the SwiGLU product
 * is computed in FP32 and h keeps its BF16 rounding): g and u accumulate in
 * double and round to FP32, silu(g) = g / (1 + e^-g) in double, the product
 * rounds to FP32 and then to BF16.  x [n, d], wg / wu [F, d] BF16 bits,
 * h [n, F] BF16 bits. */
int oracle_swiglu_bf16(const uint16_t *x, int64_t n, int32_t d, int32_t F, const uint16_t *wg,
                       const uint16_t *wu, uint16_t *h) {
  if (n < 0 || d <= 0 || F <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const uint16_t *xr = x + i * d;
    for (int32_t f = 0; f < F; ++f) {
      double ga = 0.0, ua = 0.0;
      const uint16_t *gr = wg + (int64_t)f * d;
      const uint16_t *ur = wu + (int64_t)f * d;
      for (int32_t j = 0; j < d; ++j) {
        ga += bf16_value(xr[j]) * bf16_value(gr[j]);
        ua += bf16_value(xr[j]) * bf16_value(ur[j]);
      }
      const double g = (double)(float)ga;
      const double u = (double)(float)ua;
      const double silu = g / (1.0 + exp(-g));
      h[i * F + f] = bf16_round((float)(silu * u));
    }
  }
  return 0;
}

int oracle_experts_bf16(const uint16_t *x, int64_t T, int32_t d, int32_t F,
                        int32_t k, int32_t E, const int32_t *idx, const float *w,
                        const uint16_t *const *wg, const uint16_t *const *wu,
                        const uint16_t *const *wd, const int64_t *tokens,
                        int64_t n_tokens, uint16_t *out, double *out_exact) {
  weights_t W;
  memset(&W, 0, sizeof W);
  W.wg = wg;
  W.wu = wu;
  W.wd = wd;
  return experts_impl(x, T, d, F, k, E, idx, w, &W, tokens, n_tokens, out, out_exact);
}

/* NVFP4 experts ([SGL] Highlights: "ModelOpt NVFP4" checkpoints; [VLLM]:
 * the 256 routed experts are NVFP4).  Each weight is the exact product
 * E2M1 code x E4M3 block scale x FP32 global scale.  act_quant = 1 also
 * quantises both GEMM inputs (x along d, the FP32 SwiGLU product along F) to
 * NVFP4 with the per-16 rule of nvfp4_block_roundtrip (the "quantization"
 * step of the NVFP4 MoE path, vLLM post, section "The fused graph");
 * act_quant = 0 keeps BF16 activations exactly as in the BF16 path;
 * act_quant = 2 is the 16-bit-activation reading on F16 tensor-core operands
 * [reading]: x rounded to F16 (exact inside F16's normal range) and the FP32
 * SwiGLU product rounded to F16 instead of BF16, both saturating at 65504. */
int oracle_experts_nvfp4(const uint16_t *x, int64_t T, int32_t d, int32_t F,
                         int32_t k, int32_t E, const int32_t *idx, const float *w,
                         const uint8_t *const *qg, const uint8_t *const *sfg, const float *gsg,
                         const uint8_t *const *qu, const uint8_t *const *sfu, const float *gsu,
                         const uint8_t *const *qd, const uint8_t *const *sfd, const float *gsd,
                         int32_t act_quant, const int64_t *tokens, int64_t n_tokens,
                         uint16_t *out, double *out_exact) {
  weights_t W;
  memset(&W, 0, sizeof W);
  W.qg = qg; W.sfg = sfg; W.gsg = gsg;
  W.qu = qu; W.sfu = sfu; W.gsu = gsu;
  W.qd = qd; W.sfd = sfd; W.gsd = gsd;
  W.fp4 = 1;
  W.act_quant = act_quant;
  return experts_impl(x, T, d, F, k, E, idx, w, &W, tokens, n_tokens, out, out_exact);
}

/* Dynamic FP8 experts (the pages list a compressed-tensors dynamic FP8
 * checkpoint beside the BF16 and NVFP4 ones: SGLang post, sections
 * "Highlights" and "BF16, NVFP4 and FP8 Model Support"; HF release post,
 * sections "专家混合" and "硬件要求").  [reading] The FP8 scheme is the usual dynamic one:
 * E4M3 weights with one FP32 scale per output row (each weight is exactly
 * code x scale); with act_quant != 0 both GEMM inputs are quantised per row
 * at run time with fp8_row_quantize -- x per token along d, and h per
 * (token, expert) row along F after its BF16 rounding (h is BF16 between
 * the GEMMs in every path).  act_quant = 0 keeps BF16 activations exactly as
 * in the BF16 path.  Everything else (FP32 accumulators and SwiGLU product,
 * weighted FP64 sum, one BF16 rounding) is the BF16 path's. */
int oracle_experts_fp8(const uint16_t *x, int64_t T, int32_t d, int32_t F,
                       int32_t k, int32_t E, const int32_t *idx, const float *w,
                       const uint8_t *const *qg, const float *const *sg,
                       const uint8_t *const *qu, const float *const *su,
                       const uint8_t *const *qd, const float *const *sd,
                       int32_t act_quant, const int64_t *tokens, int64_t n_tokens,
                       uint16_t *out, double *out_exact) {
  weights_t W;
  memset(&W, 0, sizeof W);
  W.eg = qg; W.seg = sg;
  W.eu = qu; W.seu = su;
  W.ed = qd; W.sed = sd;
  W.fp8 = 1;
  W.act_quant = act_quant;
  return experts_impl(x, T, d, F, k, E, idx, w, &W, tokens, n_tokens, out, out_exact);
}

/* The same layer with FP8 activations, also reporting its near ties (see
 * fp8_h_ties): tie_slack [T, d] receives, per output, the sum over the
 * token's near-tie h codes of |w * (code change) * W_d[., f]|, which is how
 * far that output moves if any subset of those codes takes the neighbouring
 * BF16 value's code; scale_tie [T] flags tokens with a row whose amax
 * element sits at such a midpoint. */
int oracle_experts_fp8_ties(const uint16_t *x, int64_t T, int32_t d, int32_t F,
                            int32_t k, int32_t E, const int32_t *idx, const float *w,
                            const uint8_t *const *qg, const float *const *sg,
                            const uint8_t *const *qu, const float *const *su,
                            const uint8_t *const *qd, const float *const *sd,
                            double tie_rel, const int64_t *tokens, int64_t n_tokens,
                            uint16_t *out, double *out_exact, double *tie_slack,
                            uint8_t *scale_tie) {
  if (!tie_slack || !scale_tie || !(tie_rel >= 0.0)) return -1;
  weights_t W;
  memset(&W, 0, sizeof W);
  W.eg = qg; W.seg = sg;
  W.eu = qu; W.seu = su;
  W.ed = qd; W.sed = sd;
  W.fp8 = 1;
  W.act_quant = 1;
  W.tie_rel = tie_rel;
  W.tie_slack = tie_slack;
  W.scale_tie = scale_tie;
  return experts_impl(x, T, d, F, k, E, idx, w, &W, tokens, n_tokens, out, out_exact);
}

/* The activation rule of the FP8 path on n rows of `cols` BF16 values:
 * codes [n, cols] and one FP32 scale per row. */
int oracle_fp8_quantize_rows(const uint16_t *x, int64_t n, int32_t cols, uint8_t *q,
                             float *scale) {
  if (n < 0 || cols <= 0) return -1;
  float *tmp = (float *)malloc(sizeof(float) * (size_t)cols);
  if (!tmp) return -3;
  for (int64_t i = 0; i < n; ++i) {
    for (int32_t j = 0; j < cols; ++j) tmp[j] = (float)bf16_value(x[i * cols + j]);
    fp8_row_quantize(tmp, cols, q + i * cols, scale + i, NULL);
  }
  free(tmp);
  return 0;
}

/* MXFP8 experts (the pages name MXFP8 beside FP8 as a precision Beam runs
 * in: vLLM post, the SkyRL paragraphs, "MXFP8 RL are supported out of the
 * box").  [reading] OCP MX format with E4M3 elements: each weight is exactly
 * code x 2^(scale - 127), one E8M0 scale per 32 consecutive elements along
 * K.  With act_quant != 0 both GEMM inputs are MX blocks too (mx_block_quantize):
 * x per 32 along d from its BF16 values, and the FP32 SwiGLU product per 32
 * along F as it is (the quantisation happens where h is produced, as in the
 * NVFP4 path).  act_quant = 0 keeps BF16 activations exactly as in the BF16
 * path.  With tie_slack / scale_tie given (act_quant != 0 only) the near
 * ties of the h quantisation are reported as for the FP8 path. */
int oracle_experts_mxfp8(const uint16_t *x, int64_t T, int32_t d, int32_t F,
                         int32_t k, int32_t E, const int32_t *idx, const float *w,
                         const uint8_t *const *qg, const uint8_t *const *sg,
                         const uint8_t *const *qu, const uint8_t *const *su,
                         const uint8_t *const *qd, const uint8_t *const *sd,
                         int32_t act_quant, double tie_rel, const int64_t *tokens,
                         int64_t n_tokens, uint16_t *out, double *out_exact, double *tie_slack,
                         uint8_t *scale_tie) {
  if ((tie_slack != NULL) != (scale_tie != NULL)) return -1;
  if (tie_slack && (!act_quant || !(tie_rel >= 0.0))) return -1;
  weights_t W;
  memset(&W, 0, sizeof W);
  W.mg = qg; W.smg = sg;
  W.mu = qu; W.smu = su;
  W.md = qd; W.smd = sd;
  W.mx = 1;
  W.act_quant = act_quant;
  W.tie_rel = tie_rel;
  W.tie_slack = tie_slack;
  W.scale_tie = scale_tie;
  return experts_impl(x, T, d, F, k, E, idx, w, &W, tokens, n_tokens, out, out_exact);
}

/* The MX activation rule on a row of n values (n % 32 == 0): E4M3 codes and
 * one E8M0 scale code per 32. */
int oracle_mx_quantize(const float *v, int64_t n, uint8_t *q, uint8_t *sc) {
  if (n < 0 || n % 32) return -1;
  for (int64_t b = 0; b < n / 32; ++b) mx_block_quantize(v + 32 * b, 32, sc + b, q + 32 * b, NULL);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* The sublayer boundary after the MoE branch                                */
/* ------------------------------------------------------------------------ */

/* One token's boundary after the MoE branch, [VLLM] "MoE and residual
 * stream" (sandwich norm: an RMSNorm after every sublayer and one before the
 * next; depth-scaled residual: the n-th add is h <- sqrt((n-1)/n) h + x/sqrt(n))
 * and "Agent-driven optimization" item 1 (post-norm, scaled residual add and
 * next pre-norm as one step, FP32 math, BF16 rounding points); [SGL]
 * "Sandwich Normalization and Depth-Scaled Residuals" (both scaled operands
 * are rounded to BF16 before the addition).  Per token, with m the layer's
 * BF16 output and h the BF16 residual stream:
 *   p  = bf16( m * g_post / sqrt(mean(m^2) + eps) )
 *   a  = bf16( c_h * h ),   b = bf16( c_x * p )
 *   h' = bf16( a + b )
 *   x  = bf16( h' * g_pre / sqrt(mean(h'^2) + eps) )
 * [reading] c_h = fp32(sqrt((n-1)/n)) and c_x = fp32(1/sqrt(n)) are given;
 * the arithmetic is FP64 with one rounding at each point listed. */
int oracle_boundary(const uint16_t *m, const uint16_t *h, const uint16_t *g_post,
                    const uint16_t *g_pre, int64_t T, int32_t d, double eps, float c_h,
                    float c_x, uint16_t *h_out, uint16_t *x_out) {
  if (T < 0 || d <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const uint16_t *mt = m + t * d, *ht = h + t * d;
    uint16_t *ho = h_out + t * d, *xo = x_out + t * d;
    double ss = 0.0;
    for (int32_t i = 0; i < d; ++i) ss += bf16_value(mt[i]) * bf16_value(mt[i]);
    const double r = 1.0 / sqrt(ss / d + eps);
    double ss2 = 0.0;
    for (int32_t i = 0; i < d; ++i) {
      const uint16_t p = bf16_round_double(bf16_value(mt[i]) * bf16_value(g_post[i]) * r);
      const uint16_t a = bf16_round_double((double)c_h * bf16_value(ht[i]));
      const uint16_t b = bf16_round_double((double)c_x * bf16_value(p));
      ho[i] = bf16_round_double(bf16_value(a) + bf16_value(b));
      ss2 += bf16_value(ho[i]) * bf16_value(ho[i]);
    }
    const double r2 = 1.0 / sqrt(ss2 / d + eps);
    for (int32_t i = 0; i < d; ++i)
      xo[i] = bf16_round_double(bf16_value(ho[i]) * bf16_value(g_pre[i]) * r2);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Scalar entry points for the pins.                                         */
/* ------------------------------------------------------------------------ */
double oracle_e2m1_value(uint8_t code) { return e2m1_value(code); }
double oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }
double oracle_e8m0_value(uint8_t code) { return e8m0_value(code); }
uint8_t oracle_e2m1_encode(float v) { return e2m1_encode(v); }
uint8_t oracle_e4m3_encode(float v) { return e4m3_encode(v); }
uint16_t oracle_bf16_round(float v) { return bf16_round(v); }
uint16_t oracle_bf16_round_double(double v) { return bf16_round_double(v); }
double oracle_f16_round(double v) { return f16_round_value(v); }

/* NVFP4 activation quantiser on a row of n values (n % 16 == 0): packed codes
 * (low nibble = even index) and one E4M3 scale per 16. */
int oracle_nvfp4_quantize(const float *v, int64_t n, uint8_t *q, uint8_t *sf) {
  if (n < 0 || n % 16) return -1;
  for (int64_t b = 0; b < n / 16; ++b) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float a = fabsf(v[b * 16 + i]);
      if (a > amax) amax = a;
    }
    sf[b] = e4m3_encode(amax / 6.0f);
    float scale = (float)e4m3_value(sf[b]);
    for (int i = 0; i < 16; i += 2) {
      uint8_t lo = scale > 0.0f ? e2m1_encode(v[b * 16 + i] / scale) : 0;
      uint8_t hi = scale > 0.0f ? e2m1_encode(v[b * 16 + i + 1] / scale) : 0;
      q[(b * 16 + i) / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
