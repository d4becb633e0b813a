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

// Split-K partial sums for small batches, register-tiled: a CTA takes 32
// experts x 16 tokens x one K chunk, each warp 4 experts of the 16 tokens.
// The CTA's chunk of W_r (32 rows) and of x (16 rows) come into shared memory
// by 16-byte asynchronous copies from every thread (many small copies: a bulk
// copy per row would queue 48 operations on the SM's copy engine), and each
// lane keeps 4 x 16 accumulators, so
// a W_r float4 serves 16 tokens and each x value (one 8-byte shared load for 4
// elements) 4 experts.  The arithmetic is that of router_partial_kernel: lane
// j adds the chunk's float4 groups j, j + 32, ... in order, each group's four
// products in order, and the 32 lane sums of a logit meet in warp_sum's
// xor-butterfly order (the butterfly of a transposing reduction, after which
// lane l holds logit l of a block of 32), so the partial sums are the same
// bits.  Optionally the CTAs of the first expert group also write the FP8 (or,
// act4, E2M1) codes of their x chunk, the activation quantiser of the layer's
// small-batch path.
struct RouterTileParams {
  const uint16_t* x;  // [T][H] bf16
  int T, H, E, kc;    // kc = H / ks elements per K chunk
  const float* W;     // [E][H]
  float* part;        // [ks][T][E]
  uint8_t* xq;        // codes of x [T][H] (act4: [T][H/2]) or null
  uint8_t* xs;        // scale bytes [T][H/32]
  int act4;
};

constexpr int kRtWarps = 8, kRtEW = 4, kRtTT = 16;
constexpr int kRtExperts = kRtWarps * kRtEW;  // 32 W_r rows per CTA
// K chunks up to this many elements are staged (32 rows of fp32 + 16 of bf16:
// 160 KB at 1024); longer chunks (a hidden size whose 128-element chunks split
// into few K chunks) take router_partial_kernel, which reads from global memory
// and forms the same sums.
constexpr int kRtMaxChunk = 1024;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

__global__ void __launch_bounds__(kRtWarps * 32, 1) router_tile_kernel(const __grid_constant__ RouterTileParams p) {
  extern __shared__ __align__(16) uint8_t rt_smem[];
  float* wsm = reinterpret_cast<float*>(rt_smem);                   // [32][kc]
  uint16_t* xsm = reinterpret_cast<uint16_t*>(wsm + kRtExperts * p.kc);  // [16][kc]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * kRtTT, nt = min(kRtTT, p.T - t0);
  const int c = blockIdx.z, k0 = c * p.kc, kc4 = p.kc / 4;
  const int eg = blockIdx.x * kRtExperts, ne = min(kRtExperts, p.E - eg);
  // W_r does not depend on the previous kernel: its copies go out first
  for (int i = threadIdx.x; i < ne * kc4; i += blockDim.x) {
    const int e = i / kc4, g = i - e * kc4;
    cp_async16(wsm + (size_t)e * p.kc + 4 * g, p.W + (size_t)(eg + e) * p.H + k0 + 4 * g);
  }
  pdl_wait();  // x may come from the previous kernel
  const int kc8 = p.kc / 8;
  for (int i = threadIdx.x; i < nt * kc8; i += blockDim.x) {
    const int t = i / kc8, g = i - t * kc8;
    cp_async16(xsm + (size_t)t * p.kc + 8 * g, p.x + (size_t)(t0 + t) * p.H + k0 + 8 * g);
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  pdl_trigger();  // the next kernel may start its prologue; it waits for all of this
  if (p.xq) {
    // the codes of x for this chunk: 8 values per thread, a quad of lanes per
    // 32-block, the blocks spread over the chunk's expert-group CTAs (one
    // trip count per quad, so a quad stays together)
    const unsigned quad = 0xFu << (lane & ~3);
    const int n32 = nt * kc8 / 4;
    const uint4* x8 = reinterpret_cast<const uint4*>(xsm);
    for (int b = blockIdx.x + gridDim.x * (int)(threadIdx.x >> 2); b < n32; b += gridDim.x * (int)(blockDim.x >> 2)) {
      const int i = 4 * b + (lane & 3);
      const int t = i / kc8, g = i - t * kc8;
      const size_t gi = (size_t)(t0 + t) * (p.H / 8) + (size_t)c * kc8 + g;  // 8-value group of x
      int ex;
      if (p.act4)
        reinterpret_cast<uint32_t*>(p.xq)[gi] = quant4(x8[i], quad, &ex);
      else
        reinterpret_cast<uint2*>(p.xq)[gi] = quant8(x8[i], quad, &ex);
      if ((lane & 3) == 0) p.xs[gi >> 2] = (uint8_t)(ex + 127);
    }
  }
  const int el = warp * kRtEW;  // the warp's first expert within the CTA
  if (el >= ne) return;         // warp-uniform; no barrier follows
  float acc[kRtEW][kRtTT];
#pragma unroll
  for (int ee = 0; ee < kRtEW; ++ee)
#pragma unroll
    for (int i = 0; i < kRtTT; ++i) acc[ee][i] = 0.f;
  const float4* w4 = reinterpret_cast<const float4*>(wsm);
  const uint2* x2 = reinterpret_cast<const uint2*>(xsm);  // 4 bf16 per element
  for (int g = lane; g < kc4; g += 32) {
    float4 wv[kRtEW];
#pragma unroll
    for (int ee = 0; ee < kRtEW; ++ee) wv[ee] = w4[min(el + ee, ne - 1) * kc4 + g];
#pragma unroll
    for (int i = 0; i < kRtTT; ++i) {
      if (i < nt) {
        const uint2 xv = x2[i * kc4 + g];
        const float xa = __uint_as_float(xv.x << 16), xb = __uint_as_float(xv.x & 0xFFFF0000u);
        const float xc = __uint_as_float(xv.y << 16), xd = __uint_as_float(xv.y & 0xFFFF0000u);
#pragma unroll
        for (int ee = 0; ee < kRtEW; ++ee) {
          acc[ee][i] = fmaf(wv[ee].x, xa, acc[ee][i]);
          acc[ee][i] = fmaf(wv[ee].y, xb, acc[ee][i]);
          acc[ee][i] = fmaf(wv[ee].z, xc, acc[ee][i]);
          acc[ee][i] = fmaf(wv[ee].w, xd, acc[ee][i]);
        }
      }
    }
  }
  // Two transposing reductions (tokens 0-7, then 8-15): at offset o the lanes
  // with bit o set keep the upper half of their items, the others the lower
  // half, each adding its partner's value of the items it keeps (own +
  // partner, as warp_sum); lane l ends with item l = 8 * ee + i.
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (8 * h >= nt) break;  // uniform
    float v[32];
#pragma unroll
    for (int ee = 0; ee < kRtEW; ++ee)
#pragma unroll
      for (int i = 0; i < 8; ++i) v[ee * 8 + i] = acc[ee][8 * h + i];
#pragma unroll
    for (int o = 16, n = 32; o > 0; o >>= 1, n >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float keep = up ? v[i + n / 2] : v[i];
        const float give = up ? v[i] : v[i + n / 2];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, o);
      }
    }
    const int ee = lane >> 3, i = 8 * h + (lane & 7);
    if (i < nt && el + ee < ne) p.part[((size_t)c * p.T + t0 + i) * p.E + eg + el + ee] = v[0];
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

bool router_tile_quantises(int H) { return H / router_ksplit(H) <= kRtMaxChunk; }

cudaError_t launch_router_tile(const uint16_t* x, int T, int H, int E, const float* W, float* part,
                               uint8_t* xq, uint8_t* xs, bool act4, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int ks = router_ksplit(H);
  if (H / ks > kRtMaxChunk) {
    if (xq) return cudaErrorInvalidValue;  // the caller quantises x itself
    const int gx = (E + kRouterWarps - 1) / kRouterWarps;
    cudaError_t le = T <= 2 ? launch_pdl(router_partial_kernel<2>, dim3(gx, (T + 1) / 2, ks), dim3(kRouterWarps * 32), 0,
                                         st, x, T, H, E, H / ks, W, part)
                            : launch_pdl(router_partial_kernel<8>, dim3(gx, (T + 7) / 8, ks), dim3(kRouterWarps * 32), 0,
                                         st, x, T, H, E, H / ks, W, part);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
  }
  RouterTileParams p{x, T, H, E, H / ks, W, part, xq, xs, act4 ? 1 : 0};
  const size_t smem = (size_t)(H / ks) * (kRtExperts * sizeof(float) + kRtTT * sizeof(uint16_t));
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(router_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kRtMaxChunk * (kRtExperts * (int)sizeof(float) + kRtTT * (int)sizeof(uint16_t)));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const dim3 grid((E + kRtExperts - 1) / kRtExperts, (T + kRtTT - 1) / kRtTT, ks);
  cudaError_t le = launch_pdl(router_tile_kernel, grid, dim3(kRtWarps * 32), smem, st, p);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

cudaError_t launch_router_split(const uint16_t* x, int T, int H, int E, int k, const float* W,
                                const float* b, const Scoring& sg, float* part, float* logits_out,
                                int32_t* idx, float* w, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int ks = router_ksplit(H);
  cudaError_t e = launch_router_tile(x, T, H, E, W, part, nullptr, nullptr, false, st);
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
