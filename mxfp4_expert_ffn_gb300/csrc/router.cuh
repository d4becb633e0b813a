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

namespace moe {

// acc[i] += sum over h in [k0, k0 + kc) of W[h] * x_i[h] for one W_r row (fp32)
// and nt <= TT bf16 tokens; lane l takes the float4 groups l, l + 32, ... in
// increasing order (so the sum order is fixed), and the row's float4 loads of a
// lane are issued in batches of 8 before they are used.  x(i, h) returns the
// two bf16 of token i at elements h, h+1 packed in a uint32 (low = h).
template <int TT, typename XFn>
__device__ __forceinline__ void router_dot(const float* __restrict__ wrow, int kc, int nt, int lane,
                                           XFn x, float (&acc)[TT]) {
  constexpr int U = 8;
  const float4* wr = reinterpret_cast<const float4*>(wrow);
  const int kc4 = kc / 4;
  for (int b = lane; b < kc4; b += 32 * U) {
    float4 wv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) wv[u] = b + 32 * u < kc4 ? __ldg(wr + b + 32 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < U; ++u) {
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

__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// The k selected (value, expert) pairs in rank order -> idx[t][r] and
// w[t][r] = exp(v_r - v_0) / sum_r' exp(v_r' - v_0), summed in rank order.
__device__ __forceinline__ void topk_softmax_write(const float* sv, const int* si, int t, int k,
                                                   int32_t* __restrict__ idx, float* __restrict__ w) {
  const float m = sv[0];
  float den = 0.f;
  for (int r = 0; r < k; ++r) den += expf(sv[r] - m);
  for (int r = 0; r < k; ++r) {
    idx[(size_t)t * k + r] = si[r];
    w[(size_t)t * k + r] = expf(sv[r] - m) / den;
  }
}

// k rounds of a warp arg-max over (value desc, index asc) on the 16 values
// per lane (v[i] is expert lane + 32 i), then the softmax over the k chosen.
__device__ __forceinline__ void select_topk(const float (&v)[16], int t, int E, int k, int lane,
                                            int32_t* __restrict__ idx, float* __restrict__ w) {
  uint32_t taken = 0;
  float sv[8];
  int si[8];
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && ranks_before(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (ranks_before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    sv[r] = bv;
    si[r] = bi;
  }
  if (lane == 0) topk_softmax_write(sv, si, t, k, idx, w);
}

}  // namespace moe
