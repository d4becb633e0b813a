// One launch that prepares a small batch (T <= 64 tokens) for the tensor-core
// expert GEMM: router logits and top-k (or the caller's routing), the FP8
// codes of x by token and the expert segments.
//
// Router: l = W_r x + b in fp32 with ties to the lower expert index and a
// softmax over the selected logits (the gate as a discrete top-6 switch:
// ai.rs, "What remains is the reference rounding itself"; llama.cpp
// discussion #28766, "Correctness").  Activations: the checkpoint's dynamic
// per-32 FP8 scheme with UE8M0 scales (FreeToken issue #444, "Is the
// quantization already supported").
//
// Phases, with no CTA ever waiting for another:
//   1. every CTA: router partial sums of (32 experts, 8 tokens, one K chunk)
//      and a share of the x quantisation;
//   2. the last CTA of each 8-token block to finish adds the K chunks of its
//      tokens' logits in a fixed order, selects top-k and writes the weights;
//   3. the last token block to finish builds the expert segments (with one
//      warp's match and ballot operations when there are at most 32 slots).
// "Last" is decided by an acquire-release atomic counter; the finisher resets
// the counter, so the next launch starts from zero.  The sums
// are the same fixed-order sums as the split-K router kernels, so the logits
// are bit-identical to theirs.
#include "common.cuh"
#include "internal.h"
#include "segments.cuh"
#include "router.cuh"

namespace moe {
namespace {

constexpr int kPrepWarps = 32;  // experts per CTA (one warp each)
constexpr int kPrepTT = 8;      // tokens per block
constexpr int kPrepTTSel = 4;   // tokens per block when the partial sums are given (9-64
                                // tokens: selection only, so more blocks sum fewer logits)

struct PrepParams {
  const uint16_t* x;
  int T, H, E, k, ns, bn;
  int route;             // 1: compute logits and top-k; 0: idx and w are given
  int parts_ready;       // route: the partial sums and the codes of x come from router_tile_kernel
  const float* W;        // [E][H] router weights (route)
  const float* b;        // [E] bias or null
  int ks;                // K chunks of the router
  float* part;           // [ks][T][E] partial sums
  float* logits_out;     // [T][E] or null
  int32_t* idx;          // [T][k] written (route) or read
  float* w;              // [T][k] written (route)
  int32_t* counters;     // [token blocks + 1], zero between launches
  Scoring sg;            // how the weights follow from the logits
  int act4;              // x codes as packed E2M1 (the FP4-activation variant)
  Workspace ws;
};

__global__ void __launch_bounds__(1024) prep_kernel(const __grid_constant__ PrepParams p) {
  pdl_wait();     // x may come from the previous kernel
  pdl_trigger();  // the expert GEMM may start its prologue; it waits for all of this
  extern __shared__ int32_t sm[];
  __shared__ int last;
  __shared__ int32_t sid_s[32];  // tiny batches: the slot ids for the segments
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // at most 32 slots, each expert's in one token tile, one token block
  const bool tiny = p.T * p.k <= 32 && p.T <= p.bn && gridDim.y == 1;

  // ---- 1a. router partial sums: warp = expert, CTA = (expert group, token block, K chunk);
  // the warp's first batch of W_r loads is in flight while the CTA's x chunk
  // (8 tokens x H/ks) is staged in shared memory
  if (p.route && !p.parts_ready) {
    const int e = blockIdx.x * kPrepWarps + warp;
    const int t0 = blockIdx.y * kPrepTT, nt = min(kPrepTT, p.T - t0);
    const int kc = p.H / p.ks, k0 = blockIdx.z * kc;
    const float* wrow = p.W + (size_t)(e < p.E ? e : 0) * p.H + k0;
    float4 wv[kRouterBatch];
    if (e < p.E) router_load_batch(reinterpret_cast<const float4*>(wrow), kc / 4, lane, wv);
    uint32_t* xsm = reinterpret_cast<uint32_t*>(sm);  // [nt][kc / 2] bf16 pairs
    for (int i = threadIdx.x; i < nt * (kc / 8); i += blockDim.x) {
      const int t = i / (kc / 8), c = i - t * (kc / 8);
      reinterpret_cast<uint4*>(xsm)[i] = *reinterpret_cast<const uint4*>(p.x + (size_t)(t0 + t) * p.H + k0 + 8 * c);
    }
    __syncthreads();
    if (e < p.E) {
      float acc[kPrepTT];
#pragma unroll
      for (int i = 0; i < kPrepTT; ++i) acc[i] = 0.f;
      auto xf = [&](int i, int h) { return xsm[i * (kc / 2) + h / 2]; };
      router_fma_batch<kPrepTT>(wv, kc / 4, lane, nt, xf, acc);
      router_dot_rest<kPrepTT>(wrow, kc, nt, lane, xf, acc);
#pragma unroll
      for (int i = 0; i < kPrepTT; ++i) {
        const float s = warp_sum(acc[i]);
        if (lane == 0 && i < nt) p.part[((size_t)blockIdx.z * p.T + t0 + i) * p.E + e] = s;
      }
    }
  }

  // ---- 1b. FP8 codes of x by token, 8 values per thread, spread over all CTAs,
  // and the zeroing of the GEMMs' arrival counters (off the serial segments)
  {
    const int cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    const int stride = gridDim.x * gridDim.y * gridDim.z * blockDim.x;
    for (int i = cta * blockDim.x + threadIdx.x; i < p.ws.split_cnt_n; i += stride) p.ws.split_cnt[i] = 0;
    for (int i = cta * blockDim.x + threadIdx.x; i < p.ws.comb_cnt_n; i += stride) p.ws.comb_cnt[i] = 0;
    const int n8 = p.parts_ready ? 0 : p.T * (p.H / 8);  // a multiple of 4: whole quads stay in or out
    const unsigned quad = 0xFu << (lane & ~3);
    const uint4* x8 = reinterpret_cast<const uint4*>(p.x);
    uint2* q8 = reinterpret_cast<uint2*>(p.ws.xq);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(p.ws.xq);
    for (int i = cta * blockDim.x + threadIdx.x; i < n8; i += stride) {
      int ex;
      if (p.act4)
        q4[i] = quant4(x8[i], quad, &ex);
      else
        q8[i] = quant8(x8[i], quad, &ex);
      if ((lane & 3) == 0) p.ws.xs[i >> 2] = (uint8_t)(ex + 127);
    }
  }

  // ---- 2. the last CTA of this token block selects its tokens' experts
  // (one acquire-release atomic per CTA: it publishes the CTA's writes, which
  // the barrier made its own, and the last arriver acquires everyone's)
  __syncthreads();
  if (gridDim.x * gridDim.z > 1) {  // (alone in its token block, a CTA is its last)
    if (threadIdx.x == 0) {
      last = atomic_add_acq_rel(&p.counters[blockIdx.y], 1) == (int)(gridDim.x * gridDim.z) - 1;
      if (last) p.counters[blockIdx.y] = 0;
    }
    __syncthreads();
    if (!last) return;
  }
  if (p.route) {
    // every thread: logits, then their selection codes and scores (so the
    // selecting warp only compares)
    const int tb = p.parts_ready ? kPrepTTSel : kPrepTT;
    const int t0 = blockIdx.y * tb, nt = min(tb, p.T - t0);
    uint32_t* okey = reinterpret_cast<uint32_t*>(sm);             // [nt][E]
    float* osc = reinterpret_cast<float*>(sm) + kPrepTT * p.E;    // [nt][E]
    for (int i = threadIdx.x; i < nt * p.E; i += blockDim.x) {
      const int t = i / p.E, e = i - t * p.E;
      // the bias is part of the logit for softmax scoring, of the selection key for sigmoid
      const float f = router_sum_partials(p.part, p.ks, p.T, p.E, t0 + t, e, p.sg.sigmoid ? nullptr : p.b);
      if (p.logits_out) p.logits_out[(size_t)(t0 + t) * p.E + e] = f;
      float kv, sv;
      topk_key_one(f, e, p.sg, kv, sv);
      okey[i] = order_key(kv);
      osc[i] = sv;
    }
    __syncthreads();
    if (warp < nt) {
      uint32_t ok[16];
      float sc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int e = lane + 32 * i;
        ok[i] = e < p.E ? okey[warp * p.E + e] : 0u;
        sc[i] = e < p.E ? osc[warp * p.E + e] : 0.f;
      }
      const int pick = select_topk_codes(ok, sc, t0 + warp, p.k, lane, p.sg, p.idx, p.w);
      if (tiny && lane < p.k) sid_s[(t0 + warp) * p.k + lane] = pick;
    }
  } else if (tiny && (int)threadIdx.x < p.T * p.k) {
    sid_s[threadIdx.x] = p.idx[threadIdx.x];
  }

  // ---- 3. the last token block builds the expert segments
  __syncthreads();
  if (gridDim.y > 1) {
    if (threadIdx.x == 0) {
      last = atomic_add_acq_rel(&p.counters[gridDim.y], 1) == (int)gridDim.y - 1;
      if (last) p.counters[gridDim.y] = 0;
    }
    __syncthreads();
    if (!last) return;
  }
  if (tiny)
    segments_tiny(sid_s, p.T, p.k, p.E, p.ns, p.ws);
  else if (p.T * p.k <= (int)blockDim.x)
    segments_small_cta(p.idx, p.T, p.k, p.E, p.ns, p.bn, p.ws, sm, false);
  else
    segments_cta(p.idx, p.T, p.k, p.E, p.ns, p.bn, p.ws, sm, false, false);
}

size_t prep_smem_bytes(int E, int H) {
  const size_t seg = (size_t)(36 * E + 2 * 4 + 1) * sizeof(int32_t), lg = (size_t)2 * kPrepTT * E * sizeof(float);
  const size_t xs = (size_t)kPrepTT * H * sizeof(uint16_t);  // bound for one K chunk of x
  const size_t small = (size_t)(4 * E + 2 * 4 + 1024 + 1) * sizeof(int32_t);  // segments_small_cta
  size_t m = seg > lg ? seg : lg;
  m = m > xs ? m : xs;
  return m > small ? m : small;
}

}  // namespace

cudaError_t prepare_prep_kernel(int E, int H) {
  return cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)prep_smem_bytes(E, H));
}

cudaError_t launch_prep(const uint16_t* x, int T, int H, int E, int k, int ns, int bn,
                        const float* W, const float* b, const Scoring& sg, float* logits_out,
                        int32_t* idx, float* w, bool route, bool act4, const Workspace& ws,
                        cudaStream_t st, bool parts_ready) {
  if (T <= 0 || T > kPrepMaxTokens) return cudaErrorInvalidValue;
  PrepParams p;
  p.x = x;
  p.T = T;
  p.H = H;
  p.E = E;
  p.k = k;
  p.ns = ns;
  p.bn = bn;
  p.route = route ? 1 : 0;
  p.parts_ready = route && parts_ready ? 1 : 0;
  p.W = W;
  p.b = b;
  p.ks = router_ksplit(H);
  p.part = ws.rpart;
  p.logits_out = logits_out;
  p.idx = idx;
  p.w = w;
  p.counters = ws.prep_cnt;
  p.sg = sg;
  p.act4 = act4 ? 1 : 0;
  p.ws = ws;
  dim3 grid;
  if (p.parts_ready) {
    grid = dim3(1, (T + kPrepTTSel - 1) / kPrepTTSel, 1);
  } else if (route) {
    grid = dim3((E + kPrepWarps - 1) / kPrepWarps, (T + kPrepTT - 1) / kPrepTT, p.ks);
  } else {
    const int n8 = T * (H / 8);
    int g = (n8 + 1023) / 1024;
    grid = dim3(g < 1 ? 1 : (g > 64 ? 64 : g), 1, 1);
  }
  { cudaError_t le_ = launch_pdl(prep_kernel, grid, dim3(1024), prep_smem_bytes(E, H), st, p); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

}  // namespace moe
