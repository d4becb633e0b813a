// Router pieces shared by the router kernels: the per-warp fp32 partial dot
// product of W_r rows with bf16 tokens, and the top-k selection with ties to
// the lower expert index and a softmax over the selected logits.  The gate is
// a discrete switch (ai.rs, "What remains is the reference rounding itself";
// llama.cpp discussion #28766, "Correctness"), so the selection is exact given
// the fp32 logits, and every kernel that computes logits adds the same
// products in the same order.
#pragma once

#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

// e^x in fp32 from IEEE operations only (Cody-Waite reduction by ln 2, split
// in two parts as the SLEEF vector math library publishes for single precision,
// a degree-7 Taylor polynomial on |r| <= ln2/2, exact scaling by 2^n), so that any
// implementation doing the same operations gets the same bits.  x is clamped
// to [-87, 88]; error a few ulp.
__device__ __forceinline__ float exp_poly_f32(float x) {
  x = fminf(fmaxf(x, -87.0f), 88.0f);
  const float n = rintf(__fmul_rn(x, 1.44269504f));
  float r = __fmaf_rn(n, -0.693145752f, x);
  r = __fmaf_rn(n, -1.42860677e-06f, r);
  float q = 1.98412698e-04f;
  q = __fmaf_rn(q, r, 1.38888889e-03f);
  q = __fmaf_rn(q, r, 8.33333333e-03f);
  q = __fmaf_rn(q, r, 4.16666667e-02f);
  q = __fmaf_rn(q, r, 1.66666667e-01f);
  q = __fmaf_rn(q, r, 0.5f);
  q = __fmaf_rn(q, r, 1.0f);
  q = __fmaf_rn(q, r, 1.0f);
  return __fmul_rn(q, __int_as_float(((int)n + 127) << 23));
}

// sigmoid(l) = 1 / (1 + e^-l), correctly rounded add and divide.
__device__ __forceinline__ float sigmoid_f32(float l) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_poly_f32(-l)));
}

// acc[i] += sum over h in [k0, k0 + kc) of W[h] * x_i[h] for one W_r row (fp32)
// and nt <= TT bf16 tokens; lane l takes the float4 groups l, l + 32, ... in
// increasing order (so the sum order is fixed), and the row's float4 loads of a
// lane are issued in batches of kRouterBatch before they are used.  x(i, h)
// returns the two bf16 of token i at elements h, h+1 packed in a uint32 (low = h).
constexpr int kRouterBatch = 8;

// The batch of float4 groups b, b + 32, ... of a row (zeros past kc4 groups).
__device__ __forceinline__ void router_load_batch(const float4* __restrict__ wr, int kc4, int b,
                                                  float4 (&wv)[kRouterBatch]) {
#pragma unroll
  for (int u = 0; u < kRouterBatch; ++u)
    wv[u] = b + 32 * u < kc4 ? __ldg(wr + b + 32 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
}

template <int TT, typename XFn>
__device__ __forceinline__ void router_fma_batch(const float4 (&wv)[kRouterBatch], int kc4, int b, int nt, XFn x,
                                                 float (&acc)[TT]) {
#pragma unroll
  for (int u = 0; u < kRouterBatch; ++u) {
    const int h4 = b + 32 * u;
    if (h4 < kc4) {
#pragma unroll
      for (int i = 0; i < TT; ++i) {
        if (i < nt) {
          const uint32_t x01 = x(i, 4 * h4), x23 = x(i, 4 * h4 + 2);
          acc[i] = fmaf(wv[u].x, __uint_as_float(x01 << 16), acc[i]);
          acc[i] = fmaf(wv[u].y, __uint_as_float(x01 & 0xFFFF0000u), acc[i]);
          acc[i] = fmaf(wv[u].z, __uint_as_float(x23 << 16), acc[i]);
          acc[i] = fmaf(wv[u].w, __uint_as_float(x23 & 0xFFFF0000u), acc[i]);
        }
      }
    }
  }
}

// The batches after the first one (already loaded into wv and added by the caller).
template <int TT, typename XFn>
__device__ __forceinline__ void router_dot_rest(const float* __restrict__ wrow, int kc, int nt, int lane, XFn x,
                                                float (&acc)[TT]) {
  const float4* wr = reinterpret_cast<const float4*>(wrow);
  const int kc4 = kc / 4;
  for (int b = lane + 32 * kRouterBatch; b < kc4; b += 32 * kRouterBatch) {
    float4 wv[kRouterBatch];
    router_load_batch(wr, kc4, b, wv);
    router_fma_batch<TT>(wv, kc4, b, nt, x, acc);
  }
}

template <int TT, typename XFn>
__device__ __forceinline__ void router_dot(const float* __restrict__ wrow, int kc, int nt, int lane,
                                           XFn x, float (&acc)[TT]) {
  float4 wv[kRouterBatch];
  router_load_batch(reinterpret_cast<const float4*>(wrow), kc / 4, lane, wv);
  router_fma_batch<TT>(wv, kc / 4, lane, nt, x, acc);
  router_dot_rest<TT>(wrow, kc, nt, lane, x, acc);
}

// The logit of (token t, expert e) from ks <= 8 K-chunk partials
// part[s][t][e], added in chunk order, plus the bias; all loads in flight.
__device__ __forceinline__ float router_sum_partials(const float* __restrict__ part, int ks, int T, int E,
                                                     int t, int e, const float* __restrict__ b) {
  float pv[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) pv[s] = s < ks ? __ldcg(part + ((size_t)s * T + t) * E + e) : 0.f;
  float f = 0.f;
#pragma unroll
  for (int s = 0; s < 8; ++s)
    if (s < ks) f += pv[s];
  return f + (b ? b[e] : 0.f);
}

// Order-preserving map of a non-NaN float key to an unsigned integer, with
// -0 and +0 mapped alike (they compare equal as floats, so the lower expert
// index decides between them).  Every key maps above 0, which marks "not a
// candidate".
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_key_value(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Selection key and score of one logit l of expert e < E: softmax keys are l
// (NaN as -infinity); sigmoid keys are sigmoid(l) + bias (NaN as -infinity),
// scores sigmoid(l).
__device__ __forceinline__ void topk_key_one(float l, int e, const Scoring& sg, float& kv, float& sv) {
  kv = -INFINITY;
  sv = 0.f;
  if (!isnan(l)) {  // a NaN logit: key -infinity, score 0
    if (sg.sigmoid) {
      sv = sigmoid_f32(l);
      kv = __fadd_rn(sv, sg.sel_bias ? sg.sel_bias[e] : 0.f);
      if (isnan(kv)) kv = -INFINITY;
    } else {
      kv = sv = l;
    }
  }
}

// Per-lane selection keys and scores from the logits l[e] of one token held by
// lane e % 32 (e = lane + 32 i); experts past E get key -infinity, score 0.
__device__ __forceinline__ void topk_keys(const float (&l)[16], int E, int lane, const Scoring& sg,
                                          float (&key)[16], float (&sc)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = lane + 32 * i;
    key[i] = -INFINITY;
    sc[i] = 0.f;
    if (e < E) topk_key_one(l[i], e, sg, key[i], sc[i]);
  }
}

// k rounds of a warp arg-max over (key desc, index asc) on the 16 keys per
// lane (key[i] is expert lane + 32 i), given as order-preserving codes ok[i]
// (order_key of the key; 0 for experts past E): the largest key by an integer
// warp reduction of the codes, then the lowest index holding it by a second
// one.  Lane r < k ends with the r-th pick and writes idx[t][r] and its
// weight: softmax w_r = exp(v_r - v_0) / sum_r' exp(v_r' - v_0) with v the
// logits; sigmoid w_r = s_r / sum_r' s_r' with s the sigmoid scores; both sums
// in rank order; then times the routed scale.  Returns the lane's pick (-1 for
// lanes >= k).
__device__ __forceinline__ int select_topk_codes(uint32_t (&ok)[16], const float (&sc)[16], int t, int k,
                                                 int lane, const Scoring& sg, int32_t* __restrict__ idx,
                                                 float* __restrict__ w) {
  int my_i = -1;
  float my_v = 0.f, my_s = 0.f;
  for (int r = 0; r < k; ++r) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = max(m, ok[i]);
    const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, m);
    unsigned cand = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 15; i >= 0; --i)
      if (ok[i] == wm) cand = (unsigned)(lane + 32 * i);
    const int wi = (int)__reduce_min_sync(0xFFFFFFFFu, cand);
    float s_w = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (lane + 32 * i == wi) {
        ok[i] = 0u;
        s_w = sc[i];
      }
    if (sg.sigmoid) s_w = __shfl_sync(0xFFFFFFFFu, s_w, wi & 31);  // the winner's score
    if (lane == r) {
      my_i = wi;
      my_v = order_key_value(wm);
      my_s = s_w;
    }
  }
  // weights: every lane forms the same rank-order sum, lane r < k its own term
  float wr;
  if (sg.sigmoid) {
    float den = 0.f;
    for (int r = 0; r < k; ++r) den = __fadd_rn(den, __shfl_sync(0xFFFFFFFFu, my_s, r));
    wr = __fmul_rn(__fdiv_rn(my_s, den), sg.scale);
  } else {
    const float m0 = __shfl_sync(0xFFFFFFFFu, my_v, 0);
    const float ex = lane < k ? expf(my_v - m0) : 0.f;
    float den = 0.f;
    for (int r = 0; r < k; ++r) den += __shfl_sync(0xFFFFFFFFu, ex, r);
    wr = (ex / den) * sg.scale;
  }
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_i;
    w[(size_t)t * k + lane] = wr;
  }
  return my_i;
}

__device__ __forceinline__ int select_topk(const float (&key)[16], const float (&sc)[16], int t, int E, int k,
                                           int lane, const Scoring& sg, int32_t* __restrict__ idx,
                                           float* __restrict__ w) {
  uint32_t ok[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) ok[i] = lane + 32 * i < E ? order_key(key[i]) : 0u;
  return select_topk_codes(ok, sc, t, k, lane, sg, idx, w);
}

}  // namespace moe
