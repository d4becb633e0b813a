// Router: fp32 logits l = W_r x + b, then per-token top-k with ties to the
// lower expert index and a softmax over the selected logits.
//
// The gate is a discrete switch (ai.rs, "What remains is the reference
// rounding itself"; llama.cpp discussion #28766, "Correctness": 6th-to-7th
// margin about 1 %), so the selection is exact given the fp32 logits.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "router.cuh"

namespace moe {
namespace {

constexpr int kRouterWarps = 8;

// One warp per (expert, group of TT tokens).  Lanes stride over H four
// elements at a time: a float4 of the expert's row and four bf16 per token.
template <int TT>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_logits_kernel(const uint16_t* __restrict__ x, int T, int H, int E,
                         const float* __restrict__ W, const float* __restrict__ b,
                         float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterWarps + warp;
  if (e >= E) return;
  const int t0 = blockIdx.y * TT;
  const int nt = min(TT, T - t0);
  float acc[TT];
#pragma unroll
  for (int i = 0; i < TT; ++i) acc[i] = 0.f;
  const uint32_t* x32 = reinterpret_cast<const uint32_t*>(x);
  router_dot<TT>(W + (size_t)e * H, H, nt, lane,
                 [&](int i, int h) { return x32[((size_t)(t0 + i) * H + h) / 2]; }, acc);
  const float bias = b ? b[e] : 0.f;
#pragma unroll
  for (int i = 0; i < TT; ++i) {
    const float s = warp_sum(acc[i]);
    if (lane == 0 && i < nt) logits[(size_t)(t0 + i) * E + e] = s + bias;
  }
}

// One warp per token; lane l holds logits l, l+32, ... (E <= 512).  k rounds
// of a warp arg-max over (value desc, index asc); NaN counts as -infinity.
__global__ void topk_kernel(const float* __restrict__ logits, int T, int E, int k, Scoring sg,
                            int32_t* __restrict__ idx, float* __restrict__ w) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  float l[16], key[16], sc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = lane + 32 * i;
    l[i] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
  }
  topk_keys(l, E, lane, sg, key, sc);
  select_topk(key, sc, t, E, k, lane, sg, idx, w);
}

// Split-K variant for small T: warp = (expert, K chunk); partial sums go to
// part[ks][t][e] and are added in fixed ks order by topk_sum_kernel.
template <int TT>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_partial_kernel(const uint16_t* __restrict__ x, int T, int H, int E, int kc,
                          const float* __restrict__ W, float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterWarps + warp;
  if (e >= E) return;
  const int t0 = blockIdx.y * TT, ks = blockIdx.z;
  const int nt = min(TT, T - t0);
  float acc[TT];
#pragma unroll
  for (int i = 0; i < TT; ++i) acc[i] = 0.f;
  const int k0 = ks * kc;
  const uint32_t* x32 = reinterpret_cast<const uint32_t*>(x);
  router_dot<TT>(W + (size_t)e * H + k0, kc, nt, lane,
                 [&](int i, int h) { return x32[((size_t)(t0 + i) * H + k0 + h) / 2]; }, acc);
#pragma unroll
  for (int i = 0; i < TT; ++i) {
    const float sum = warp_sum(acc[i]);
    if (lane == 0 && i < nt) part[((size_t)ks * T + t0 + i) * E + e] = sum;
  }
}

// One CTA per token: all threads add the split-K partials of the token's
// logits (fixed ks order, plus bias) in parallel, then one warp selects.
__global__ void __launch_bounds__(256) topk_sum_kernel(const float* __restrict__ part, int ksplit,
                                                       const float* __restrict__ b, int T, int E,
                                                       int k, Scoring sg, float* __restrict__ logits_out,
                                                       int32_t* __restrict__ idx,
                                                       float* __restrict__ w) {
  pdl_wait();
  pdl_trigger();
  __shared__ float lg[512];
  const int t = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    // the bias is part of the logit for softmax scoring, of the selection key for sigmoid
    const float f = router_sum_partials(part, ksplit, T, E, t, e, sg.sigmoid ? nullptr : b);
    lg[e] = f;
    if (logits_out) logits_out[(size_t)t * E + e] = f;
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float l[16], key[16], sc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = lane + 32 * i;
    l[i] = e < E ? lg[e] : -INFINITY;
  }
  topk_keys(l, E, lane, sg, key, sc);
  select_topk(key, sc, t, E, k, lane, sg, idx, w);
}

}  // namespace

int router_ksplit(int H) {
  const int chunks = H / 128;
  for (int ks = 8; ks > 1; --ks)
    if (chunks % ks == 0) return ks;
  return 1;
}

cudaError_t launch_router_split(const uint16_t* x, int T, int H, int E, int k, const float* W,
                                const float* b, const Scoring& sg, float* part, float* logits_out,
                                int32_t* idx, float* w, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int ks = router_ksplit(H);
  const int gx = (E + kRouterWarps - 1) / kRouterWarps;
  if (T <= 2)
    { cudaError_t le_ = launch_pdl(router_partial_kernel<2>, dim3(dim3(gx, (T + 1) / 2, ks)), dim3(kRouterWarps * 32), 0, st, x, T, H, E, H / ks, W, part); if (le_ != cudaSuccess) return le_; }
  else
    { cudaError_t le_ = launch_pdl(router_partial_kernel<8>, dim3(dim3(gx, (T + 7) / 8, ks)), dim3(kRouterWarps * 32), 0, st, x, T, H, E, H / ks, W, part); if (le_ != cudaSuccess) return le_; }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  { cudaError_t le_ = launch_pdl(topk_sum_kernel, dim3(T), dim3(256), 0, st, part, ks, b, T, E, k, sg, logits_out, idx, w); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_topk_sum(const float* part, int ksplit, const float* b, int T, int E, int k,
                            const Scoring& sg, float* logits_out, int32_t* idx, float* w,
                            cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  { cudaError_t le_ = launch_pdl(topk_sum_kernel, dim3(T), dim3(256), 0, st, part, ksplit, b, T, E, k, sg, logits_out, idx, w); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_router_logits(const uint16_t* x, int T, int H, int E, const float* W,
                                 const float* b, float* logits, int num_sms, cudaStream_t st) {
  (void)num_sms;
  if (T == 0) return cudaSuccess;
  const int gx = (E + kRouterWarps - 1) / kRouterWarps;
  if (T <= 2) {
    { cudaError_t le_ = launch_pdl(router_logits_kernel<2>, dim3(dim3(gx, (T + 1) / 2)), dim3(kRouterWarps * 32), 0, st, x, T, H, E, W, b,
                                                                                logits); if (le_ != cudaSuccess) return le_; }
  } else {
    { cudaError_t le_ = launch_pdl(router_logits_kernel<8>, dim3(dim3(gx, (T + 7) / 8)), dim3(kRouterWarps * 32), 0, st, x, T, H, E, W, b,
                                                                                logits); if (le_ != cudaSuccess) return le_; }
  }
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, const Scoring& sg, int32_t* idx,
                        float* w, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  { cudaError_t le_ = launch_pdl(topk_kernel, dim3((T + 7) / 8), dim3(256), 0, st, logits, T, E, k, sg, idx, w); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

}  // namespace moe
