/*
 * CPU oracle for the routed MXFP4 mixture-of-experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only tests/, the smoke check in __graft_entry__.py and the
 * cpu_baseline / reference leg of bench.py use it.  It shares no code, header,
 * table or helper with the CUDA library; every table below is built from the
 * format's definition.
 *
 * Plain and slow on purpose: fp64 arithmetic, values decoded one element at a
 * time, no blocking or reordering.  Rounding happens only where the layer
 * definition puts it: the FP8 codes of x and of h, the fp32 router logits and
 * the final bf16 output.
 *
 * Sources (web pages, by title and section):
 *  - FreeToken issue #444 "[Model] DeepSeek-V4.1-Flash (deepseek_v41)",
 *    section "Is the quantization already supported": FP4 routed experts, FP8
 *    dense, dynamic activation scheme, UE8M0 scale format.
 *  - same issue, "Architecture delta vs deepseek_v4": 384 routed + 1 shared
 *    experts, top-6, gate/up/down = 3 x 5120 x 2304 FP4 per expert.
 *  - same issue, janit's comment item 2 "Routed expert bytes per token":
 *    packed E2M1 codes with one E8M0 scale per 32 elements ("ds_fp4").
 *  - ai.rs "DeepSeek-V4.1-Flash on an RTX 5090", "What remains is the reference
 *    rounding itself": the MoE gate is a discrete switch over the top-6
 *    scores; the shared expert sees the same input and arithmetic.
 *  - llama.cpp discussion #28766, "Correctness": top-6 choices, 6th-to-7th
 *    margin about 1 %.
 * Where the pages are silent (scoring function, SwiGLU form, scale rule,
 * tie order) the readings are listed with each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ formats */

/* E2M1 (OCP MX FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * Magnitudes of codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign,
 * so code 8 is -0. */
double orc_e2m1_value(int code) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[code & 7];
  return (code & 8) ? -v : v;
}

/* UE8M0: an unsigned biased exponent, value 2^(s-127); 255 is NaN. */
double orc_ue8m0_value(int s) {
  if (s == 255) return NAN;
  return ldexp(1.0, s - 127);
}

/* E4M3 (the FN variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, largest finite 448, smallest subnormal
 * 2^-9. */
double orc_e4m3_value(int code) {
  int sign = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);          /* m/8 * 2^(1-7) */
  else
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -v : v;
}

/* Nearest finite E4M3 value, ties to the even code, saturating at 448: an
 * exhaustive search over the 127 non-negative finite codes.  The sign is kept
 * for every input, so a negative value that rounds to zero gives 0x80. */
int orc_e4m3_encode(double v) {
  int sign = signbit(v) ? 1 : 0;
  double a = fabs(v);
  int best = 0;
  double bestd = INFINITY;
  if (isnan(v)) return 0x7F;
  for (int c = 0; c <= 0x7E; ++c) {
    double d = fabs(orc_e4m3_value(c) - a);
    if (d < bestd || (d == bestd && (c % 2) == 0)) {
      best = c;
      bestd = d;
    }
  }
  return (sign << 7) | best;
}

/* The block exponent of the dynamic FP8 scheme: the smallest integer e with
 * amax <= 448 * 2^e, limited to [-127, 127] so that e + 127 is a UE8M0 byte;
 * an all-zero block takes e = 0.  (Reading: the pages fix the UE8M0 scale
 * format and the dynamic scheme but not the rule; this one never saturates.) */
int orc_block_exponent(double amax) {
  int e = -127;
  if (amax == 0.0) return 0;
  while (e < 127 && amax > ldexp(448.0, e)) ++e;
  return e;
}

/* Quantise n values (one block) to E4M3 codes with a shared UE8M0 scale. */
void orc_quantize_block(const double* v, int n, uint8_t* q, uint8_t* s) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  int e = orc_block_exponent(amax);
  *s = (uint8_t)(e + 127);
  for (int i = 0; i < n; ++i) q[i] = (uint8_t)orc_e4m3_encode(ldexp(v[i], -e));
}

double orc_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to bf16 (8 significant bits), nearest, ties to even. */
uint16_t orc_bf16_round(double v) {
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v), r;
  if (isnan(v)) return 0x7FC0;
  if (a == 0.0) {
    r = 0.0;
  } else if (a < 0x1p-126) {
    r = rint(ldexp(a, 133)) * 0x1p-133; /* subnormal spacing 2^-133 */
  } else {
    int E;
    frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    r = ldexp(rint(ldexp(a, 8 - E)), E - 8);
  }
  uint32_t u;
  if (r > 0x1.FCp127) {
    u = 0x7F800000u;
  } else {
    float f = (float)r; /* exact: r is a bf16 value */
    memcpy(&u, &f, 4);
  }
  return (uint16_t)((u >> 16) | ((uint32_t)neg << 15));
}

/* Dynamic per-32 FP8 quantisation of bf16 activations x[T][H] into codes
 * q[T][H] and scale bytes s[T][H/32] (FreeToken issue #444, "Is the
 * quantization already supported": activation_scheme dynamic, scale_fmt
 * ue8m0; block of 32 as for the experts' scales). */
void orc_quantize_act(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s) {
  double blk[32];
  for (int t = 0; t < T; ++t)
    for (int b = 0; b < H / 32; ++b) {
      for (int i = 0; i < 32; ++i) blk[i] = orc_bf16_value(x[(size_t)t * H + b * 32 + i]);
      orc_quantize_block(blk, 32, q + (size_t)t * H + b * 32, s + (size_t)t * (H / 32) + b);
    }
}

/* ------------------------------------------------- FP4 activations (variant) */
/* The FP4-activation variant quantises x and h to E2M1 per 32 with a UE8M0
 * scale instead of E4M3 (reading: the same dynamic block rule with the E2M1
 * maximum 6 in place of 448; the pages measure FP4-block activation error as
 * large, so this stays an option).  Finite inputs only. */

/* Nearest E2M1 value, ties to the even code, saturating at 6: an exhaustive
 * search over the eight non-negative codes.  The sign is kept for every input,
 * so a negative value that rounds to zero gives code 8. */
int orc_e2m1_encode(double v) {
  int sign = signbit(v) ? 1 : 0;
  double a = fabs(v);
  int best = 0;
  double bestd = INFINITY;
  if (a > 6.0) return (sign << 3) | 7;
  for (int c = 0; c <= 7; ++c) {
    double d = fabs(orc_e2m1_value(c) - a);
    if (d < bestd || (d == bestd && (c % 2) == 0)) {
      best = c;
      bestd = d;
    }
  }
  return (sign << 3) | best;
}

/* The block exponent of the FP4 variant: the smallest integer e with
 * amax <= 6 * 2^e, limited to [-127, 127]; an all-zero block takes e = 0. */
int orc_block_exponent4(double amax) {
  int e = -127;
  if (amax == 0.0) return 0;
  while (e < 127 && amax > ldexp(6.0, e)) ++e;
  return e;
}

/* Quantise n values (one block) to E2M1 codes (one per byte, 0..15) with a
 * shared UE8M0 scale. */
void orc_quantize_block4(const double* v, int n, uint8_t* q, uint8_t* s) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  int e = orc_block_exponent4(amax);
  *s = (uint8_t)(e + 127);
  for (int i = 0; i < n; ++i) q[i] = (uint8_t)orc_e2m1_encode(ldexp(v[i], -e));
}

/* Per-32 FP4 quantisation of bf16 activations x[T][H] into packed codes
 * q[T][H/2] (element 2i in the low nibble of byte i, as the weights) and
 * scale bytes s[T][H/32]. */
void orc_quantize_act4(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s) {
  double blk[32];
  uint8_t c[32];
  for (int t = 0; t < T; ++t)
    for (int b = 0; b < H / 32; ++b) {
      for (int i = 0; i < 32; ++i) blk[i] = orc_bf16_value(x[(size_t)t * H + b * 32 + i]);
      orc_quantize_block4(blk, 32, c, s + (size_t)t * (H / 32) + b);
      for (int i = 0; i < 16; ++i)
        q[(size_t)t * (H / 2) + b * 16 + i] = (uint8_t)(c[2 * i] | (c[2 * i + 1] << 4));
    }
}

/* ------------------------------------------------------------------ routing */

/* Router logits l[t][e] = sum_h x[t][h] * W[e][h] + b[e], in fp64, then
 * rounded to fp32.  b may be NULL. */
void orc_router_logits(const uint16_t* x, int T, int H, int E, const float* W, const float* b,
                       float* logits, int nthreads) {
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
#endif
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += orc_bf16_value(x[(size_t)t * H + h]) * (double)W[(size_t)e * H + h];
      if (b) acc += (double)b[e];
      logits[(size_t)t * E + e] = (float)acc;
    }
  (void)nthreads;
}

typedef struct {
  double key;
  int index;
} orc_scored;

/* Selection order: larger score first, equal scores by lower expert index.
 * NaN scores rank as -infinity.  +0 and -0 are equal. */
static int orc_rank_cmp(const void* pa, const void* pb) {
  const orc_scored* a = (const orc_scored*)pa;
  const orc_scored* b = (const orc_scored*)pb;
  if (a->key > b->key) return -1;
  if (a->key < b->key) return 1;
  return (a->index < b->index) ? -1 : (a->index > b->index);
}

/* Top-k of each token's fp32 logits by a full sort, then the combine weights
 * as a softmax over the k selected logits (equal to renormalising the
 * full softmax over the selected experts).  Slot j of token t holds the
 * rank-j expert. */
void orc_topk(const float* logits, int T, int E, int k, int32_t* idx, double* w) {
  orc_scored* a = (orc_scored*)malloc(sizeof(orc_scored) * (size_t)E);
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double v = (double)logits[(size_t)t * E + e];
      a[e].key = isnan(v) ? -INFINITY : v;
      a[e].index = e;
    }
    qsort(a, (size_t)E, sizeof(orc_scored), orc_rank_cmp);
    double m = a[0].key, den = 0.0;
    for (int j = 0; j < k; ++j) den += exp(a[j].key - m);
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = a[j].index;
      w[(size_t)t * k + j] = exp(a[j].key - m) / den;
    }
  }
  free(a);
}

/* --------------------------------------------------------- sigmoid scoring */

/* A second router scoring (DeepSeek-V3 style; the pages never name the score
 * function, see the readings): s = sigmoid(l) of the unbiased logit, the bias
 * added to s for the selection only, weights s / (sum of the k selected s),
 * times a routed scaling factor.  Which experts are selected is decided in
 * fp32, the precision the layer computes it in, so sigmoid here is a fixed
 * sequence of correctly rounded fp32 operations: e^x by Cody and Waite's
 * reduction x = n ln2 + r (n = round-half-even(x log2 e), ln 2 split into
 * 0.693145752 + 1.42860677e-6 so that n * 0.693145752 is exact -- the same
 * two-part split of ln 2 that the SLEEF vector math library publishes for
 * single precision), e^r by its
 * degree-7 Taylor polynomial in Horner form with fused multiply-adds
 * (truncation below 6e-9 relative on |r| <= ln2/2), then times 2^n; x is first
 * clamped to [-87, 88].  Compiled without floating-point contraction. */
float orc_exp_f32(float x) {
  x = fminf(fmaxf(x, -87.0f), 88.0f);
  const float n = rintf(x * 1.44269504f);
  float r = fmaf(n, -0.693145752f, x);
  r = fmaf(n, -1.42860677e-06f, r);
  float q = 1.98412698e-04f;  /* 1/7! */
  q = fmaf(q, r, 1.38888889e-03f);  /* 1/6! */
  q = fmaf(q, r, 8.33333333e-03f);  /* 1/5! */
  q = fmaf(q, r, 4.16666667e-02f);  /* 1/4! */
  q = fmaf(q, r, 1.66666667e-01f);  /* 1/3! */
  q = fmaf(q, r, 0.5f);
  q = fmaf(q, r, 1.0f);
  q = fmaf(q, r, 1.0f);
  const uint32_t bits = (uint32_t)((int)n + 127) << 23;
  float p2;
  memcpy(&p2, &bits, sizeof p2);
  return q * p2;
}

float orc_sigmoid_f32(float l) { return 1.0f / (1.0f + orc_exp_f32(-l)); }

/* Sigmoid top-k: key_e = fp32(s_e + bias_e) (NaN logits: key -infinity,
 * s = 0), selection by (key desc, index asc) with a full sort, weights in
 * fp64: w_j = s_j / sum_j' s_j' * scale, j in rank order. */
void orc_topk_sigmoid(const float* logits, const float* bias, int T, int E, int k, double scale,
                      int32_t* idx, double* w) {
  orc_scored* a = (orc_scored*)malloc(sizeof(orc_scored) * (size_t)E);
  float* sc = (float*)malloc(sizeof(float) * (size_t)E);
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      const float l = logits[(size_t)t * E + e];
      if (isnan(l)) {
        sc[e] = 0.0f;
        a[e].key = -INFINITY;
      } else {
        sc[e] = orc_sigmoid_f32(l);
        const float key = sc[e] + (bias ? bias[e] : 0.0f);
        a[e].key = isnan(key) ? -INFINITY : (double)key;
      }
      a[e].index = e;
    }
    qsort(a, (size_t)E, sizeof(orc_scored), orc_rank_cmp);
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += (double)sc[a[j].index];
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = a[j].index;
      w[(size_t)t * k + j] = (double)sc[a[j].index] / den * scale;
    }
  }
  free(sc);
  free(a);
}

/* Expert segments of the T*k slots (slot s = t*k + j): off[e] = number of
 * slots routed to experts below e (off[E] = T*k); perm lists the slots
 * expert by expert, each expert's slots in increasing slot order. */
void orc_segments(const int32_t* idx, int T, int k, int E, int32_t* off, int32_t* perm) {
  int S = T * k, p = 0;
  for (int e = 0; e < E; ++e) {
    off[e] = p;
    for (int s = 0; s < S; ++s)
      if (idx[s] == e) perm[p++] = s;
  }
  off[E] = p;
}

/* ------------------------------------------------------------------ experts */

/* A weight matrix with N output rows and K inputs, in one of two formats:
 *  fmt 0 (MXFP4, every expert by default): codes [N][K/2], two E2M1 per byte,
 *        low nibble = even k, high nibble = odd k; scales [N][K/32] UE8M0, one per
 *        row and 32 inputs;
 *  fmt 1 (FP8 with 32 x 32 blocks, the shared-expert variant): codes [N][K] E4M3;
 *        scales [N/32][K/32] UE8M0, one per block of 32 rows x 32 inputs -- the
 *        checkpoint's dense-layer scheme (FreeToken issue #444, "Is the quantization
 *        already supported": quant_method fp8, weight_block_size [32, 32],
 *        scale_fmt ue8m0; ai.rs, "The defect that never raised an error": the
 *        fp8 scale block is 32 x 32). */
typedef struct {
  const uint8_t* codes;
  const uint8_t* scales;
  int fmt;
} orc_mat;

typedef struct {
  orc_mat gate, up, down; /* gate/up: N = I, K = H; down: N = H, K = I */
} orc_expert;

/* The 256 UE8M0 values, filled from orc_ue8m0_value when the library loads
 * (a lookup instead of an ldexp per weight; same values). */
static double orc_ue8m0_table[256];
__attribute__((constructor)) static void orc_fill_tables(void) {
  for (int s = 0; s < 256; ++s) orc_ue8m0_table[s] = orc_ue8m0_value(s);
}

/* Element (r, c) of a weight matrix with K columns. */
static double orc_mx_weight(const orc_mat* m, int K, int r, int c) {
  if (m->fmt == 1)
    return orc_e4m3_value(m->codes[(size_t)r * K + c]) *
           orc_ue8m0_table[m->scales[(size_t)(r / 32) * (K / 32) + c / 32]];
  uint8_t byte = m->codes[(size_t)r * (K / 2) + c / 2];
  int code = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
  return orc_e2m1_value(code) * orc_ue8m0_table[m->scales[(size_t)r * (K / 32) + c / 32]];
}

/* One activation code (one per byte) of the given format: E4M3 (act4 = 0) or
 * E2M1 (act4 = 1). */
static double orc_act_value(int act4, uint8_t code) {
  return act4 ? orc_e2m1_value(code & 15) : orc_e4m3_value(code);
}

static void orc_quantize_block_fmt(int act4, const double* v, int n, uint8_t* q, uint8_t* s) {
  if (act4)
    orc_quantize_block4(v, n, q, s);
  else
    orc_quantize_block(v, n, q, s);
}

/* One expert on one token whose activation is already quantised (one code per
 * element, E4M3 or, act4 = 1, E2M1):
 *   g = Wg x^, u = Wu x^, h = silu(g) * u = g / (1 + e^-g) * u,
 *   h quantised per 32 (same rule and format as x), o = Wd h^.
 * (Readings: SwiGLU with silu on the gate projection and no clamp; h is
 * quantised before the down projection like every activation under the
 * checkpoint's dynamic scheme.)  h_out (I), hq (I), hs (I/32) may be NULL. */
int orc_expert_ffn_fmt(const orc_expert* ex, int H, int I, int act4, const uint8_t* xq,
                       const uint8_t* xs, double* h_out, uint8_t* hq_out, uint8_t* hs_out,
                       double* o) {
  if (!ex || !ex->gate.codes || !ex->up.codes || !ex->down.codes) return -1;
  double* xh = (double*)malloc(sizeof(double) * (size_t)H);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* hh = (double*)malloc(sizeof(double) * (size_t)I);
  uint8_t* hq = (uint8_t*)malloc((size_t)I);
  uint8_t* hs = (uint8_t*)malloc((size_t)I / 32);
  for (int c = 0; c < H; ++c) xh[c] = orc_act_value(act4, xq[c]) * orc_ue8m0_value(xs[c / 32]);
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += orc_mx_weight(&ex->gate, H, i, c) * xh[c];
      u += orc_mx_weight(&ex->up, H, i, c) * xh[c];
    }
    h[i] = g / (1.0 + exp(-g)) * u;
  }
  for (int b = 0; b < I / 32; ++b) orc_quantize_block_fmt(act4, h + b * 32, 32, hq + b * 32, hs + b);
  for (int i = 0; i < I; ++i) hh[i] = orc_act_value(act4, hq[i]) * orc_ue8m0_value(hs[i / 32]);
  for (int r = 0; r < H; ++r) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += orc_mx_weight(&ex->down, I, r, i) * hh[i];
    o[r] = acc;
  }
  if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)I);
  if (hq_out) memcpy(hq_out, hq, (size_t)I);
  if (hs_out) memcpy(hs_out, hs, (size_t)I / 32);
  free(xh);
  free(h);
  free(hh);
  free(hq);
  free(hs);
  return 0;
}

/* The FP8-activation expert (the layer's definition). */
int orc_expert_ffn(const orc_expert* ex, int H, int I, const uint8_t* xq, const uint8_t* xs,
                   double* h_out, uint8_t* hq_out, uint8_t* hs_out, double* o) {
  return orc_expert_ffn_fmt(ex, H, I, 0, xq, xs, h_out, hq_out, hs_out, o);
}

/* The layer on T tokens given the routing (idx[T][k], w[T][k]):
 *   y[t] = bf16( sum_shared o_s + sum_j w[t][j] * o_{idx[t][j]} )
 * and, with a residual r, y[t] = bf16(r[t] + bf16(...)).  The shared experts
 * see every token with weight 1.  experts[e] may hold NULL pointers for
 * experts no token uses; returns -1 if a used expert is missing.
 * y64 (may be NULL) receives the sum before bf16 rounding. */
int orc_moe_layer_fmt(int T, int H, int I, int E, int k, int n_shared, int act4, const uint16_t* x,
                      const int32_t* idx, const double* w, const orc_expert* experts,
                      const orc_expert* shared, const uint16_t* residual, uint16_t* y, double* y64,
                      int nthreads) {
  int* bad = (int*)calloc((size_t)(T > 0 ? T : 1), sizeof(int));
  int status = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
#endif
  for (int t = 0; t < T; ++t) {
    uint8_t* xq = (uint8_t*)malloc((size_t)H);
    uint8_t* xs = (uint8_t*)malloc((size_t)H / 32);
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    double* acc = (double*)calloc((size_t)H, sizeof(double));
    {
      double blk[32];
      for (int b = 0; b < H / 32; ++b) {
        for (int i = 0; i < 32; ++i) blk[i] = orc_bf16_value(x[(size_t)t * H + b * 32 + i]);
        orc_quantize_block_fmt(act4, blk, 32, xq + b * 32, xs + b);
      }
    }
    for (int s = 0; s < n_shared; ++s) {
      if (orc_expert_ffn_fmt(&shared[s], H, I, act4, xq, xs, NULL, NULL, NULL, o) != 0) bad[t] = 1;
      else
        for (int r = 0; r < H; ++r) acc[r] += o[r];
    }
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      if (e < 0 || e >= E || orc_expert_ffn_fmt(&experts[e], H, I, act4, xq, xs, NULL, NULL, NULL, o) != 0) {
        bad[t] = 1;
        continue;
      }
      for (int r = 0; r < H; ++r) acc[r] += w[(size_t)t * k + j] * o[r];
    }
    for (int r = 0; r < H; ++r) {
      size_t p = (size_t)t * H + r;
      uint16_t yb = orc_bf16_round(acc[r]);
      if (residual) yb = orc_bf16_round(orc_bf16_value(residual[p]) + orc_bf16_value(yb));
      y[p] = yb;
      if (y64) y64[p] = acc[r];
    }
    free(xq);
    free(xs);
    free(o);
    free(acc);
  }
  for (int t = 0; t < T; ++t)
    if (bad[t]) status = -1;
  free(bad);
  (void)nthreads;
  return status;
}

/* The layer with FP8 activations (its definition). */
int orc_moe_layer(int T, int H, int I, int E, int k, int n_shared, const uint16_t* x,
                  const int32_t* idx, const double* w, const orc_expert* experts,
                  const orc_expert* shared, const uint16_t* residual, uint16_t* y, double* y64,
                  int nthreads) {
  return orc_moe_layer_fmt(T, H, I, E, k, n_shared, 0, x, idx, w, experts, shared, residual, y, y64,
                           nthreads);
}

/* Root-mean-square normalisation of each token row (no learned gain):
 * out = bf16(x / sqrt(mean(x^2) + eps)).  Applied to each layer's input in
 * the 8-layer stack.  (Reading: the pages leave open what lies between
 * stacked MoE layers; without a normalisation the synthetic layer's output
 * grows with the square of its input and overflows bf16 by the fifth layer.) */
void orc_rmsnorm(const uint16_t* x, int T, int H, double eps, uint16_t* out) {
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
      double v = orc_bf16_value(x[(size_t)t * H + h]);
      ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / H + eps);
    for (int h = 0; h < H; ++h)
      out[(size_t)t * H + h] = orc_bf16_round(orc_bf16_value(x[(size_t)t * H + h]) * inv);
  }
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
