// Grouped MXFP4 expert GEMV on the SIMT pipes (the decode-sized path).
//
// Streams only the experts that have tokens (active list from the segment
// pass), 16 bytes = one 32-element MX block per lane per row, dequantises in
// registers (cvt e2m1x2 -> f16x2; every E2M1 x E4M3 product is exact in fp32),
// accumulates in fp32 and applies the two UE8M0 scales once per block.
// Bank layout and per-32 scales: FreeToken issue #444, janit's comment item 2
// ("packed-e2m1 + E8M0-per-32"); expert shape 3 x 5120 x 2304: same issue,
// "Architecture delta vs deepseek_v4".
//
// ffn_up:   one work unit = (active expert, 32 consecutive rows of I); the
//           unit's gate and up rows give h = silu(g) * u for those 32 rows,
//           which is exactly one FP8 block of h, quantised in the epilogue.
// ffn_down: one work unit = (active expert, 64 consecutive rows of H);
//           writes fp32 expert outputs per position.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct MatPtr {
  const uint8_t* codes;
  const uint8_t* scales;
};

// Matrix `which` (0 gate, 1 up, 2 down) of expert id e.
__device__ __forceinline__ MatPtr expert_mat(const ExpertBank& bk, int e, int which) {
  const size_t n_up = (size_t)bk.I * bk.H;  // elements of a gate/up/down matrix
  const bool shared = e >= bk.E;
  const size_t ei = shared ? (size_t)(e - bk.E) : (size_t)e;
  const uint8_t* c;
  const uint8_t* s;
  if (which == 0) {
    c = shared ? bk.sgc : bk.gc;
    s = shared ? bk.sgs : bk.gs;
  } else if (which == 1) {
    c = shared ? bk.suc : bk.uc;
    s = shared ? bk.sus : bk.us;
  } else {
    c = shared ? bk.sdc : bk.dc;
    s = shared ? bk.sds : bk.ds;
  }
  return {c + ei * (n_up / 2), s + ei * (n_up / 32)};
}

// Dot product of one 32-element block: 16 f16x2 weights with 16 f16x2
// activations, fp32 accumulation.
__device__ __forceinline__ float block_dot(const uint32_t (&wh)[16], const uint32_t* xa) {
  float p0 = 0.f, p1 = 0.f;
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    p0 = fma2_f16_f32(wh[j], xa[j], p0);
    p1 = fma2_f16_f32(wh[j + 1], xa[j + 1], p1);
  }
  return p0 + p1;
}

__device__ __forceinline__ void decode_block(const uint4 cw, uint32_t (&wh)[16]) {
  const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    e2m1x4_to_f16x4(w4[q] & 0xFFFFu, wh[4 * q], wh[4 * q + 1]);
    e2m1x4_to_f16x4(w4[q] >> 16, wh[4 * q + 2], wh[4 * q + 3]);
  }
}

// Stages the FP8 activations of MT consecutive positions into shared memory as
// f16x2 pairs (exact) plus their block exponents.  Positions >= m stage zeros.
template <int MT>
__device__ __forceinline__ void stage_act(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                          int K, const int32_t* rowid, int m, uint32_t* xh,
                                          int* xe) {
  const int n16 = K / 16;  // 16 codes per uint4
  for (int i = threadIdx.x; i < MT * n16; i += kThreads) {
    const int tt = i / n16, j = i - tt * n16;
    uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (tt < m) {
      const uint4 c = *reinterpret_cast<const uint4*>(q + (size_t)rowid[tt] * K + 16 * j);
      const uint32_t cc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        r[2 * u] = e4m3x2_to_f16x2((uint16_t)(cc[u] & 0xFFFFu));
        r[2 * u + 1] = e4m3x2_to_f16x2((uint16_t)(cc[u] >> 16));
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(xh + (size_t)tt * (K / 2) + 8 * j);
    dst[0] = make_uint4(r[0], r[1], r[2], r[3]);
    dst[1] = make_uint4(r[4], r[5], r[6], r[7]);
  }
  for (int i = threadIdx.x; i < MT * (K / 32); i += kThreads) {
    const int tt = i / (K / 32), b = i - tt * (K / 32);
    xe[i] = tt < m ? (int)s[(size_t)rowid[tt] * (K / 32) + b] - 127 : 0;
  }
}

// 2^k as fp32 for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

template <int MT>
__global__ void __launch_bounds__(kThreads) ffn_up_simt_kernel(ExpertBank bk, Workspace ws) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  const int H = bk.H, I = bk.I;
  uint32_t* xh = reinterpret_cast<uint32_t*>(smem);          // [MT][H/2] f16x2
  int* xe = reinterpret_cast<int*>(xh + MT * (H / 2));        // [MT][H/32]
  float* hb = reinterpret_cast<float*>(xe + MT * (H / 32));   // [32][MT]
  int* rowid = reinterpret_cast<int*>(hb + 32 * MT);          // [MT]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rb = I / 32;
  const int n_units = *ws.n_active * n_rb;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int a = u / n_rb;
    const int e = ws.active[a];
    const int r0 = (u - a * n_rb) * 32;
    const int p0 = ws.off[e], m = ws.cnt[e];
    const MatPtr G = expert_mat(bk, e, 0), U = expert_mat(bk, e, 1);
    const int rw = r0 + 4 * warp;
    for (int c0 = 0; c0 < m; c0 += MT) {
      const int mt = min(MT, m - c0);
      __syncthreads();
      if (threadIdx.x < MT) rowid[threadIdx.x] = threadIdx.x < mt ? ws.pos_tok[p0 + c0 + threadIdx.x] : 0;
      __syncthreads();
      stage_act<MT>(ws.xq, ws.xs, H, rowid, mt, xh, xe);
      __syncthreads();
      float acc[8][MT];
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[r][t] = 0.f;
      for (int b = lane; b < H / 32; b += 32) {
        uint4 cw[8];
        float sc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const MatPtr& M = r < 4 ? G : U;
          const size_t row = (size_t)(rw + (r & 3));
          cw[r] = __ldg(reinterpret_cast<const uint4*>(M.codes + row * (H / 2)) + b);
          sc[r] = pow2f((int)__ldg(M.scales + row * (H / 32) + b) - 127);
        }
        uint32_t xa[MT][16];
        float xsc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const uint4* src = reinterpret_cast<const uint4*>(xh + (size_t)t * (H / 2) + 16 * b);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 q = src[v];
            xa[t][4 * v] = q.x;
            xa[t][4 * v + 1] = q.y;
            xa[t][4 * v + 2] = q.z;
            xa[t][4 * v + 3] = q.w;
          }
          xsc[t] = pow2f(xe[t * (H / 32) + b]);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          uint32_t wh[16];
          decode_block(cw[r], wh);
#pragma unroll
          for (int t = 0; t < MT; ++t) acc[r][t] = fmaf(block_dot(wh, xa[t]) * sc[r], xsc[t], acc[r][t]);
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[r][t] = warp_sum(acc[r][t]);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            const float g = acc[i][t], up = acc[4 + i][t];
            hb[(4 * warp + i) * MT + t] = g / (1.0f + expf(-g)) * up;
          }
      }
      __syncthreads();
      if (warp < mt) {
        // token `warp` of this chunk: lane i holds h of row r0 + i
        const float hv = hb[lane * MT + warp];
        const int ex = fp8_block_exponent(warp_max(fabsf(hv)));
        const uint32_t code = e4m3x2(scale_pow2_neg(hv, ex), 0.f) & 0xFFu;
        const size_t p = (size_t)(p0 + c0 + warp);
        ws.hq[p * I + r0 + lane] = (uint8_t)code;
        if (lane == 0) ws.hs[p * (I / 32) + r0 / 32] = (uint8_t)(ex + 127);
      }
    }
  }
}

template <int MT>
__global__ void __launch_bounds__(kThreads) ffn_down_simt_kernel(ExpertBank bk, Workspace ws) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  const int H = bk.H, I = bk.I;
  uint32_t* xh = reinterpret_cast<uint32_t*>(smem);          // [MT][I/2] f16x2
  int* xe = reinterpret_cast<int*>(xh + MT * (I / 2));        // [MT][I/32]
  float* ob = reinterpret_cast<float*>(xe + MT * (I / 32));   // [MT][64]
  int* rowid = reinterpret_cast<int*>(ob + 64 * MT);          // [MT]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rb = H / 64;
  const int n_units = *ws.n_active * n_rb;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int a = u / n_rb;
    const int e = ws.active[a];
    const int r0 = (u - a * n_rb) * 64;
    const int p0 = ws.off[e], m = ws.cnt[e];
    const MatPtr D = expert_mat(bk, e, 2);
    const int rw = r0 + 8 * warp;
    for (int c0 = 0; c0 < m; c0 += MT) {
      const int mt = min(MT, m - c0);
      __syncthreads();
      if (threadIdx.x < MT) rowid[threadIdx.x] = p0 + c0 + (threadIdx.x < mt ? threadIdx.x : 0);
      __syncthreads();
      stage_act<MT>(ws.hq, ws.hs, I, rowid, mt, xh, xe);
      __syncthreads();
      float acc[8][MT];
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[r][t] = 0.f;
      for (int b = lane; b < I / 32; b += 32) {
        uint4 cw[8];
        float sc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const size_t row = (size_t)(rw + r);
          cw[r] = __ldg(reinterpret_cast<const uint4*>(D.codes + row * (I / 2)) + b);
          sc[r] = pow2f((int)__ldg(D.scales + row * (I / 32) + b) - 127);
        }
        uint32_t xa[MT][16];
        float xsc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const uint4* src = reinterpret_cast<const uint4*>(xh + (size_t)t * (I / 2) + 16 * b);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 q = src[v];
            xa[t][4 * v] = q.x;
            xa[t][4 * v + 1] = q.y;
            xa[t][4 * v + 2] = q.z;
            xa[t][4 * v + 3] = q.w;
          }
          xsc[t] = pow2f(xe[t * (I / 32) + b]);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          uint32_t wh[16];
          decode_block(cw[r], wh);
#pragma unroll
          for (int t = 0; t < MT; ++t) acc[r][t] = fmaf(block_dot(wh, xa[t]) * sc[r], xsc[t], acc[r][t]);
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[r][t] = warp_sum(acc[r][t]);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int t = 0; t < MT; ++t) ob[t * 64 + 8 * warp + r] = acc[r][t];
      }
      __syncthreads();
      for (int i = threadIdx.x; i < mt * 64; i += kThreads) {
        const int t = i >> 6, j = i & 63;
        ws.o[(size_t)(p0 + c0 + t) * H + r0 + j] = ob[t * 64 + j];
      }
    }
  }
}

template <int MT>
size_t up_smem(int H) { return (size_t)MT * (H / 2) * 4 + (size_t)MT * (H / 32) * 4 + 32 * MT * 4 + MT * 4; }
template <int MT>
size_t down_smem(int I) { return (size_t)MT * (I / 2) * 4 + (size_t)MT * (I / 32) * 4 + 64 * MT * 4 + MT * 4; }

}  // namespace

// Grid: a persistent loop over (active expert, row block); sized to fill the
// GPU and capped by the largest possible number of units.
static int simt_grid(int units_max, int num_sms, int per_sm) {
  int g = num_sms * per_sm;
  return g < units_max ? g : (units_max > 0 ? units_max : 1);
}

cudaError_t prepare_ffn_simt(int H, int I) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(ffn_up_simt_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)up_smem<1>(H)))) return e;
  if ((e = cudaFuncSetAttribute(ffn_up_simt_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)up_smem<4>(H)))) return e;
  if ((e = cudaFuncSetAttribute(ffn_down_simt_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)down_smem<1>(I)))) return e;
  return cudaFuncSetAttribute(ffn_down_simt_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)down_smem<4>(I));
}

cudaError_t launch_ffn_up_simt(const ExpertBank& bank, int T, int k, int n_shared,
                               const Workspace& ws, int num_sms, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int units_max = (bank.E + n_shared) * (bank.I / 32);
  if (T == 1) {
    { cudaError_t le_ = launch_pdl(ffn_up_simt_kernel<1>, dim3(simt_grid(units_max, num_sms, 4)), dim3(kThreads), up_smem<1>(bank.H), st, bank, ws); if (le_ != cudaSuccess) return le_; }
  } else {
    { cudaError_t le_ = launch_pdl(ffn_up_simt_kernel<4>, dim3(simt_grid(units_max, num_sms, 2)), dim3(kThreads), up_smem<4>(bank.H), st, bank, ws); if (le_ != cudaSuccess) return le_; }
  }
  (void)k;
  return cudaGetLastError();
}

cudaError_t launch_ffn_down_simt(const ExpertBank& bank, int T, int k, int n_shared,
                                 const Workspace& ws, int num_sms, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int units_max = (bank.E + n_shared) * (bank.H / 64);
  if (T == 1) {
    { cudaError_t le_ = launch_pdl(ffn_down_simt_kernel<1>, dim3(simt_grid(units_max, num_sms, 4)), dim3(kThreads), down_smem<1>(bank.I), st, bank, ws); if (le_ != cudaSuccess) return le_; }
  } else {
    { cudaError_t le_ = launch_pdl(ffn_down_simt_kernel<4>, dim3(simt_grid(units_max, num_sms, 2)), dim3(kThreads), down_smem<4>(bank.I), st, bank, ws); if (le_ != cudaSuccess) return le_; }
  }
  (void)k;
  return cudaGetLastError();
}

}  // namespace moe
