// Router logits for many tokens on the tensor cores.
//
// l[t][e] = sum_h x[t][h] * W_r[e][h] with x in bf16 and W_r in fp32.  W_r is
// split once, at layer creation, into three bf16 matrices W1 + W2 + W3 (the
// top, middle and low 8 significant bits), so every product x * Wi is exact
// in fp32 and tcgen05.mma kind::f16 accumulates the three in fp32: the result
// has the accuracy of an fp32 dot product.  K is split over CTAs; the top-k
// pass adds the partial sums in fixed order and the bias.  (The router is a
// switch over the top-6 scores: ai.rs, "What remains is the reference
// rounding itself".)
//
// One CTA per SM, six warps: TMA producer, MMA issuer, four epilogue warps.
// A unit is (K split, 128 experts, 128 tokens); a stage is 64 elements of K:
// one 48 KB TMA op for the three weight parts and one 16 KB op for x.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace moe {

struct RouterParams {
  CUtensorMap w3;  // {H, E, 3} bf16, box {64, 128, 3}
  CUtensorMap x;   // {H, T} bf16, box {64, 128}
  int T, E, H, ksplit;
  float* part;     // [ksplit][T][E]
  int32_t* err;
};

namespace {

using namespace sm100;

constexpr int kRThreads = 192;
constexpr int kRStages = 3;
constexpr int kRWTile = 3 * 128 * 128;  // bytes: three parts, 128 rows x 128 bytes
constexpr int kRXTile = 128 * 128;
constexpr int kRStage = kRWTile + kRXTile;
constexpr int kRSmem = 1024 + kRStages * kRStage;
constexpr uint32_t kRWait = 1u << 24;

// kind::f16 instruction descriptor: fp32 accumulate, A = B = bf16, K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* m, int c0, int c1, int c2,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kRThreads, 1) router_mma_kernel(const __grid_constant__ RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full_bar[kRStages], empty_bar[kRStages], accf[2], acce[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_mt = (p.E + 127) / 128, n_nt = (p.T + 127) / 128;
  const int total = p.ksplit * n_mt * n_nt;
  const int kst = p.H / 64 / p.ksplit;  // stages per unit
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, 256);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_wait();  // x may come from the previous kernel
  pdl_trigger();
  auto give_up = [&]() {
    atomicOr(p.err, kErrTimeout);
    *(volatile int*)&abort_flag = 1;
  };
  auto aborted = [&]() { return *(volatile int*)&abort_flag != 0; };
  // unit u -> (ks, mt, nt), tokens innermost
  auto unit = [&](int u, int& ks, int& mt, int& nt) {
    nt = u % n_nt;
    mt = (u / n_nt) % n_mt;
    ks = u / (n_nt * n_mt);
  };

  if (warp == 0) {
    if (lane == 0) {
      uint32_t g = 0;
      int last[kRStages] = {-1, -1, -1};
      for (int u = blockIdx.x; u < total && !aborted(); u += gridDim.x) {
        int ks, mt, nt;
        unit(u, ks, mt, nt);
        for (int s = 0; s < kst; ++s, ++g) {
          const int slot = g % kRStages;
          const uint32_t ph = (g / kRStages) & 1;
          if (!mbar_wait(&empty_bar[slot], ph ^ 1, kRWait)) { give_up(); break; }
          uint8_t* st = base + slot * kRStage;
          const int k0 = (ks * kst + s) * 64;
          mbar_expect_tx(&full_bar[slot], kRStage);
          tma_3d(st, &p.w3, k0, mt * 128, 0, &full_bar[slot]);
          tma_load_2d(st + kRWTile, &p.x, k0, nt * 128, &full_bar[slot]);
          for (int i = 0; i < kRStages; ++i)
            if (i == slot) last[i] = (int)ph;
        }
      }
      for (int s = 0; s < kRStages; ++s)
        if (last[s] >= 0) mbar_wait(&full_bar[s], (uint32_t)last[s], kRWait);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t g = 0, it = 0;
      const uint32_t idesc = idesc_bf16(128, 128);
      for (int u = blockIdx.x; u < total && !aborted(); u += gridDim.x, ++it) {
        const int buf = it & 1;
        if (!mbar_wait(&acce[buf], ((it >> 1) & 1) ^ 1, kRWait)) { give_up(); break; }
        fence_after();
        bool ok = true;
        for (int s = 0; s < kst; ++s, ++g) {
          const int slot = g % kRStages;
          if (!mbar_wait(&full_bar[slot], (g / kRStages) & 1, kRWait)) { give_up(); ok = false; break; }
          fence_after();
          const uint32_t sw = smem_u32(base + slot * kRStage), sx = sw + kRWTile;
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int part = 0; part < 3; ++part)
              mma_bf16(tmem + buf * 128, sw128_desc(sw + part * 16384 + 32 * k), sw128_desc(sx + 32 * k),
                       idesc, (s | k | part) ? 1u : 0u);
          mma_commit(&empty_bar[slot]);
        }
        if (!ok) break;
        mma_commit(&accf[buf]);
      }
    }
  } else {
    const int q = warp & 3;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < total && !aborted(); u += gridDim.x, ++it) {
      int ks, mt, nt;
      unit(u, ks, mt, nt);
      const int buf = it & 1;
      if (!mbar_wait(&accf[buf], (it >> 1) & 1, kRWait)) { give_up(); break; }
      fence_after();
      const int e = mt * 128 + 32 * q + lane;
      float* out = p.part + ((size_t)ks * p.T + nt * 128) * p.E + e;
#pragma unroll 1
      for (int c = 0; c < 128; c += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + buf * 128 + c, v);
        tmem_ld_wait();
        if (c + 16 >= 128) {
          fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce[buf]);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (e < p.E && nt * 128 + c + j < p.T) out[(size_t)(c + j) * p.E] = __uint_as_float(v[j]);
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// W_r (fp32) -> three bf16 parts, w = w1 + w2 + w3 to the last bits.
__global__ void split_bf16x3_kernel(const float* __restrict__ w, size_t n, uint16_t* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 a = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(a);
    const __nv_bfloat16 b = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(b);
    const __nv_bfloat16 c = __float2bfloat16_rn(r2);
    out[i] = __bfloat16_as_ushort(a);
    out[n + i] = __bfloat16_as_ushort(b);
    out[2 * n + i] = __bfloat16_as_ushort(c);
  }
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                             CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                             CUtensorMapFloatOOBfill);

EncodeFn encode() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
    cudaGetLastError();
  }
  return fn;
}

}  // namespace

int router_mma_ksplit(int H) {
  const int chunks = H / 64;
  for (int ks = 4; ks > 1; --ks)
    if (chunks % ks == 0) return ks;
  return 1;
}

cudaError_t router_split_weights(const float* w, int E, int H, uint16_t* w3, cudaStream_t st) {
  const size_t n = (size_t)E * H;
  split_bf16x3_kernel<<<1024, 256, 0, st>>>(w, n, w3);
  return cudaGetLastError();
}

bool router_map_weights(CUtensorMap* m, const uint16_t* w3, int E, int H) {
  EncodeFn enc = encode();
  if (!enc || !w3) return false;
  cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)E, 3};
  cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)E * H * 2};
  cuuint32_t box[3] = {64, 128, 3}, es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(w3), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_router_mma(const CUtensorMap& w3map, const uint16_t* x, int T, int E, int H,
                              float* part, int32_t* err, int num_sms, cudaStream_t st) {
  RouterParams p;
  memset(&p, 0, sizeof(p));
  p.w3 = w3map;
  EncodeFn enc = encode();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  cuuint32_t box[2] = {64, 128}, es[2] = {1, 1};
  if (enc(&p.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  p.T = T;
  p.E = E;
  p.H = H;
  p.ksplit = router_mma_ksplit(H);
  p.part = part;
  p.err = err;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(router_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  { cudaError_t le_ = launch_pdl(router_mma_kernel, dim3(num_sms), dim3(kRThreads), kRSmem, st, p); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

}  // namespace moe
