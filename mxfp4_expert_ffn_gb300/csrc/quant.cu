// Activation quantisation, expert segments, combine and RMS normalisation.
//
// Quantisation: the dynamic per-32 FP8 activation scheme of the checkpoint
// (FreeToken issue #444, "Is the quantization already supported":
// activation_scheme dynamic, scale_fmt ue8m0).  Segments and combine: the
// routed MoE block (384 routed + 1 shared, top-6; same issue, "Architecture
// delta vs deepseek_v4").  All four are HBM- or latency-bound and run on the
// SIMT pipes with 128-bit accesses.
#include "common.cuh"
#include "internal.h"
#include "segments.cuh"

namespace moe {
namespace {

constexpr int kMaxPositions = 16;  // positions of one token: top-k (<= 8) + shared experts (<= 4)

// One thread per 8 bf16 values; four consecutive threads form one 32-block.
__global__ void quantize_act_kernel(const uint4* __restrict__ x, int n8, uint2* __restrict__ q,
                                    uint8_t* __restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const unsigned quad = 0xFu << (lane & ~3);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += gridDim.x * blockDim.x) {
    int e;
    q[i] = quant8(x[i], quad, &e);
    if ((lane & 3) == 0) s[i >> 2] = (uint8_t)(e + 127);
  }
}

// The FP4-activation variant of the quantiser above: 8 values -> 4 bytes.
__global__ void quantize_act4_kernel(const uint4* __restrict__ x, int n8, uint32_t* __restrict__ q,
                                     uint8_t* __restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const unsigned quad = 0xFu << (lane & ~3);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += gridDim.x * blockDim.x) {
    int e;
    q[i] = quant4(x[i], quad, &e);
    if ((lane & 3) == 0) s[i >> 2] = (uint8_t)(e + 127);
  }
}

// Large batches: the segments in two launches over many CTAs (segments.cuh).
__global__ void __launch_bounds__(1024) segments_count_kernel(const int32_t* __restrict__ idx, int T, int k,
                                                              int E, int ns, int bn, Workspace ws) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t sm[];
  segments_count_cta(idx, T, k, E, ns, bn, ws, sm);
}

__global__ void __launch_bounds__(1024) segments_place_kernel(const int32_t* __restrict__ idx, int T, int k,
                                                              int E, int ns, Workspace ws) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t sm[];
  segments_place_cta(idx, T, k, E, ns, ws, sm);
}

// The codes of x in slot order, token-major: one CTA per token quantises its
// row once and stores the codes at each of the token's positions (its valid
// routed slots, slot_pos[t*k + j], and its shared-expert positions
// S + s*T + t), so each row is read and quantised once instead of once per
// position.  Positions freed by invalid ids are not written (no tile reads
// them).  A4: packed E2M1 (4 bytes per 8 values) instead of E4M3.
template <bool A4>
__global__ void quantize_scatter_kernel(const uint16_t* __restrict__ x, int T, int H, int k, int ns,
                                        const int32_t* __restrict__ slot_pos, uint8_t* __restrict__ xg,
                                        uint8_t* __restrict__ xgs) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t pos[kMaxPositions];
  const int lane = threadIdx.x & 31;
  const unsigned quad = 0xFu << (lane & ~3);
  const int per_row = H / 8;  // a multiple of 16: whole quads stay in or out
  const size_t S = (size_t)T * k;
  const size_t row_bytes = A4 ? H / 2 : H;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();  // the previous token's positions are no longer read
    const int np = k + ns;
    if ((int)threadIdx.x < np)
      pos[threadIdx.x] = (int)threadIdx.x < k ? slot_pos[(size_t)t * k + threadIdx.x]
                                              : (int)(S + (size_t)((int)threadIdx.x - k) * T + t);
    __syncthreads();
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    for (int j = threadIdx.x; j < per_row; j += blockDim.x) {
      int e;
      uint2 c8 = make_uint2(0u, 0u);
      uint32_t c4 = 0u;
      if (A4)
        c4 = quant4(src[j], quad, &e);
      else
        c8 = quant8(src[j], quad, &e);
      for (int q = 0; q < np; ++q) {
        const int p = pos[q];
        if (p < 0) continue;  // an invalid id: the slot has no position
        if (A4)
          reinterpret_cast<uint32_t*>(xg + (size_t)p * row_bytes)[j] = c4;
        else
          reinterpret_cast<uint2*>(xg + (size_t)p * row_bytes)[j] = c8;
        if ((lane & 3) == 0) xgs[(size_t)p * (H / 32) + (j >> 2)] = (uint8_t)(e + 127);
      }
    }
  }
}

// Expert segments in one CTA of 1024 threads (segments.cuh).
__global__ void __launch_bounds__(1024) segments_kernel(const int32_t* __restrict__ idx, int T,
                                                        int k, int E, int ns, int bn, Workspace ws,
                                                        int scatter_smem) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t sm[];
  segments_cta(idx, T, k, E, ns, bn, ws, sm, scatter_smem != 0);
}

// y[t] = bf16( sum_s o[S + s*T + t] + sum_j w[t][j] * o[slot_pos[t*k + j]] ),
// accumulated in fp32 in that fixed order; optional residual added to the
// bf16-rounded sum.  Four consecutive h per thread.
// yf (expert parallelism): the fp32 sum itself, not rounded and without the
// residual, is stored (the layer's share of y, added across ranks later).
__global__ void combine_kernel(const float* __restrict__ o, const int32_t* __restrict__ slot_pos,
                               const float* __restrict__ w, int T, int H, int k, int ns,
                               const uint16_t* __restrict__ res, uint16_t* __restrict__ y,
                               float* __restrict__ yf) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;  // tokens on x: up to 2^31 - 1 of them
  const int h = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (h >= H) return;
  const size_t S = (size_t)T * k;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < ns; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(o + (S + (size_t)s * T + t) * H + h);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  for (int j = 0; j < k; ++j) {
    const int p = slot_pos[(size_t)t * k + j];
    if (p < 0) continue;
    const float wj = w[(size_t)t * k + j];
    const float4 v = *reinterpret_cast<const float4*>(o + (size_t)p * H + h);
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  }
  if (yf) {
    *reinterpret_cast<float4*>(yf + (size_t)t * H + h) = acc;
    return;
  }
  float r[4] = {acc.x, acc.y, acc.z, acc.w};
  uint16_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = __bfloat16_as_ushort(__float2bfloat16_rn(r[i]));
  if (res) {
    const uint2 rv = *reinterpret_cast<const uint2*>(res + (size_t)t * H + h);
    const uint16_t rb[4] = {(uint16_t)(rv.x & 0xFFFF), (uint16_t)(rv.x >> 16),
                            (uint16_t)(rv.y & 0xFFFF), (uint16_t)(rv.y >> 16)};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      b[i] = __bfloat16_as_ushort(
          __float2bfloat16_rn(bf16_bits_to_float(rb[i]) + bf16_bits_to_float(b[i])));
  }
  *reinterpret_cast<uint2*>(y + (size_t)t * H + h) =
      make_uint2(b[0] | ((uint32_t)b[1] << 16), b[2] | ((uint32_t)b[3] << 16));
}

// y[t] = bf16( sum over parts r = 0 .. R-1, in that order, of part[r][t] ),
// then with a residual bf16(residual[t] + y[t]): the ranks' shares of a layer
// under expert parallelism, added in a fixed order.
__global__ void combine_parts_kernel(const float* __restrict__ part, int R, int T, int H,
                                     const uint16_t* __restrict__ res, uint16_t* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int h = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (h >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < R; ++r) {
    const float4 v = *reinterpret_cast<const float4*>(part + ((size_t)r * T + t) * H + h);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const float f[4] = {acc.x, acc.y, acc.z, acc.w};
  uint16_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = __bfloat16_as_ushort(__float2bfloat16_rn(f[i]));
  if (res) {
    const uint2 rv = *reinterpret_cast<const uint2*>(res + (size_t)t * H + h);
    const uint16_t rb[4] = {(uint16_t)(rv.x & 0xFFFF), (uint16_t)(rv.x >> 16),
                            (uint16_t)(rv.y & 0xFFFF), (uint16_t)(rv.y >> 16)};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      b[i] = __bfloat16_as_ushort(
          __float2bfloat16_rn(bf16_bits_to_float(rb[i]) + bf16_bits_to_float(b[i])));
  }
  *reinterpret_cast<uint2*>(y + (size_t)t * H + h) =
      make_uint2(b[0] | ((uint32_t)b[1] << 16), b[2] | ((uint32_t)b[3] << 16));
}

// out[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps)); fixed-order block reduction.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* __restrict__ x, int H,
                                                      float eps, uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[256];
  const int t = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  float ss = 0.f;
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x) {
    const uint4 v = xr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = __uint_as_float(w[j] << 16), b = __uint_as_float(w[j] & 0xFFFF0000u);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  red[threadIdx.x] = ss;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  const float inv = 1.0f / sqrtf(red[0] / (float)H + eps);
  uint4* outr = reinterpret_cast<uint4*>(out + (size_t)t * H);
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x) {
    const uint4 v = xr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = __uint_as_float(w[j] << 16) * inv;
      const float b = __uint_as_float(w[j] & 0xFFFF0000u) * inv;
      r[j] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
    }
    // out may alias x: each thread writes only the elements it reads here, and
    // every read of the sum-of-squares pass finished before the reduction.
    outr[i] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

}  // namespace

cudaError_t launch_quantize_act(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s,
                                cudaStream_t st) {
  const int n8 = T * (H / 8);
  if (n8 == 0) return cudaSuccess;
  int blocks = (n8 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  { cudaError_t le_ = launch_pdl(quantize_act_kernel, dim3(blocks), dim3(256), 0, st, reinterpret_cast<const uint4*>(x), n8,
                                               reinterpret_cast<uint2*>(q), s); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

size_t segments_smem_bytes(int E) { return (size_t)(36 * E + 2 * 4 + 1) * sizeof(int32_t); }
constexpr size_t kSegmentsSmemMax = 200 * 1024;  // room for the position table of up to ~30k slots

// One CTA up to kSegSingleMax slots; above, two launches over up to kSegCtas CTAs.
constexpr int kSegSingleMax = 4096;
size_t segments_count_smem(int E, int ns) { return (size_t)(36 * E + 2 * ns + 2) * sizeof(int32_t); }
size_t segments_place_smem(int E) { return (size_t)32 * E * sizeof(int32_t); }

cudaError_t launch_segments(const int32_t* idx, int T, int k, int E, int n_shared, int bn,
                            const Workspace& ws, cudaStream_t st) {
  const int S = T * k;
  if (S > kSegSingleMax) {
    int G = S / 768;
    G = G < 2 ? 2 : (G > kSegCtas ? kSegCtas : G);
    { cudaError_t le_ = launch_pdl(segments_count_kernel, dim3(G), dim3(1024), segments_count_smem(E, n_shared), st, idx, T, k, E, n_shared, bn, ws); if (le_ != cudaSuccess) return le_; }
    { cudaError_t le_ = launch_pdl(segments_place_kernel, dim3(G), dim3(1024), segments_place_smem(E), st, idx, T, k, E, n_shared, ws); if (le_ != cudaSuccess) return le_; }
    return cudaGetLastError();
  }
  const size_t base = segments_smem_bytes(E), with_table = base + (size_t)T * k * sizeof(int32_t);
  const bool scatter = with_table <= kSegmentsSmemMax;  // position table in shared memory
  { cudaError_t le_ = launch_pdl(segments_kernel, dim3(1), dim3(1024), scatter ? with_table : base, st, idx, T, k, E, n_shared, bn, ws, scatter ? 1 : 0); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_quantize_scatter(const uint16_t* x, int T, int H, int k, int ns, const int32_t* slot_pos,
                                    uint8_t* xg, uint8_t* xgs, bool act4, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (k + ns > kMaxPositions) return cudaErrorInvalidValue;
  const int blocks = T < 65536 ? T : 65536;
  if (act4) {
    { cudaError_t le_ = launch_pdl(quantize_scatter_kernel<true>, dim3(blocks), dim3(256), 0, st, x, T, H, k, ns, slot_pos, xg, xgs); if (le_ != cudaSuccess) return le_; }
  } else {
    { cudaError_t le_ = launch_pdl(quantize_scatter_kernel<false>, dim3(blocks), dim3(256), 0, st, x, T, H, k, ns, slot_pos, xg, xgs); if (le_ != cudaSuccess) return le_; }
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_act4(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s,
                                 cudaStream_t st) {
  const int n8 = T * (H / 8);
  if (n8 == 0) return cudaSuccess;
  int blocks = (n8 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  { cudaError_t le_ = launch_pdl(quantize_act4_kernel, dim3(blocks), dim3(256), 0, st, reinterpret_cast<const uint4*>(x), n8,
                                 reinterpret_cast<uint32_t*>(q), s); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t prepare_segments_kernel(int E) {
  const size_t b = segments_smem_bytes(E);
  cudaError_t e = cudaFuncSetAttribute(segments_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(b > kSegmentsSmemMax ? b : kSegmentsSmemMax));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(segments_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)segments_count_smem(E, 4));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(segments_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)segments_place_smem(E));
  return e;
}

cudaError_t launch_combine(const Workspace& ws, int T, int H, int k, int n_shared, const float* w,
                           const uint16_t* residual, uint16_t* y, cudaStream_t st, float* y_f32) {
  if (T == 0) return cudaSuccess;
  dim3 grid(T, (H / 4 + 255) / 256);
  { cudaError_t le_ = launch_pdl(combine_kernel, dim3(grid), dim3(256), 0, st, ws.o, ws.slot_pos, w, T, H, k, n_shared, residual, y, y_f32); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_combine_parts(const float* part, int R, int T, int H, const uint16_t* residual, uint16_t* y,
                                 cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  dim3 grid(T, (H / 4 + 255) / 256);
  cudaError_t le = launch_pdl(combine_parts_kernel, grid, dim3(256), 0, st, part, R, T, H, residual, y);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps, uint16_t* out,
                           cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  { cudaError_t le_ = launch_pdl(rmsnorm_kernel, dim3(T), dim3(256), 0, st, x, H, eps, out); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

}  // namespace moe
