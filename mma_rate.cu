// Microbenchmark of the block-scaled tensor-core MMAs the expert GEMM uses,
// without memory traffic: cycles per tcgen05.mma with operands resident in
// shared memory (zeros) and scale factors 2^0, for kind::mxf8f6f4 (A E2M1
// expanded to a byte per element, B E4M3, K = 32, scale_vec::1X; the layer's
// kind) and kind::mxf4 (A and B packed E2M1, K = 64, scale_vec::2X; the
// FP4-activation variant's kind), M = 128 and N from 16 to 256.  One CTA per
// SM, one issuing thread; every wait is bounded.  Built and run by
// `python bench.py --mma-rates`; a measurement tool beside the benchmark, not
// part of the library.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

__device__ __forceinline__ uint32_t s32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t sw128(uint32_t a) {
  return (uint64_t)((a & 0x3FFFF) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

template <int KIND>
__global__ void __launch_bounds__(128, 1) rate(int N, int rounds, unsigned long long* cyc, int* err) {
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = sm;           // 128 rows x 128 B
  uint8_t* sB = sm + 16384;   // up to 256 rows x 128 B
  __shared__ __align__(8) uint64_t bar_done;
  __shared__ uint32_t tslot;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (16384 + 32768) / 16; i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s32(&bar_done)));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(s32(&tslot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = tslot;
  for (int c = 384; c < 512; ++c)
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tmem + ((uint32_t)(32 * warp) << 16) + c), "r"(0x7F7F7F7Fu));
  asm volatile("tcgen05.wait::st.sync.aligned;");
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  if (threadIdx.x == 0) {
    const uint32_t fa = KIND == 0 ? 5u : 1u, fb = KIND == 0 ? 0u : 1u;
    const uint32_t idesc0 = (1u << 23) | (fa << 7) | (fb << 10) | ((uint32_t)(N >> 3) << 17) | ((128u >> 4) << 24);
    const uint64_t a0 = sw128(s32(sA)), b0 = sw128(s32(sB));
    const uint32_t sfa = tmem + 384, sfb = tmem + 448;
    unsigned long long t0 = clock64();
    for (int r = 0; r < rounds; ++r) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (KIND == 0) {
          const uint32_t idesc = idesc0 | ((uint32_t)k << 4) | ((uint32_t)k << 29);
          asm volatile(
              "{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
              "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;}\n"
              ::"r"(tmem + (r & 1) * 128), "l"(a0 + 2 * k), "l"(b0 + 2 * k), "r"(idesc), "r"(1), "r"(sfa + (r & 3) * 4), "r"(sfb + (r & 1) * 8));
        } else {
          // K = 64 per instruction: 32 bytes of each packed row; scale bytes 0-1 or 2-3
          const uint32_t sid = (uint32_t)(k & 1) * 2;
          const uint32_t idesc = idesc0 | (sid << 4) | (sid << 29);
          asm volatile(
              "{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
              "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;}\n"
              ::"r"(tmem + (r & 1) * 128), "l"(a0 + 2 * k), "l"(b0 + 2 * k), "r"(idesc), "r"(1), "r"(sfa + ((k >> 1) + 2 * (r & 1)) * 4), "r"(sfb + (r & 1) * 8 + (k >> 1) * 4));
        }
      }
    }
    unsigned long long t1 = clock64();
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s32(&bar_done)) : "memory");
    bool ok = false;
    for (int it = 0; it < (1 << 24) && !ok; ++it) {
      uint32_t d;
      asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0; selp.u32 %0, 1, 0, p; }" : "=r"(d) : "r"(s32(&bar_done)) : "memory");
      ok = d != 0;
    }
    if (!ok) atomicOr(err, 1);
    unsigned long long t2 = clock64();
    cyc[blockIdx.x * 2] = t1 - t0;
    cyc[blockIdx.x * 2 + 1] = t2 - t0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

template <int KIND>
void run(int sms, unsigned long long* cyc, int* err) {
  cudaFuncSetAttribute(rate<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024);
  const int rounds = 512;  // 2048 MMAs
  for (int N : {16, 64, 112, 128, 256}) {
    unsigned long long h[2 * 1024];
    double best = 1e30;
    for (int rep = 0; rep < 3; ++rep) {
      rate<KIND><<<sms, 128, 120 * 1024>>>(N, rounds, cyc, err);
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) { printf("cuda error %s\n", cudaGetErrorString(e)); return; }
      cudaMemcpy(h, cyc, sizeof(unsigned long long) * 2 * sms, cudaMemcpyDeviceToHost);
      double mt = 0;
      for (int i = 0; i < sms; ++i) mt += h[2 * i + 1];
      mt /= sms;
      if (mt < best) best = mt;
    }
    int e = 0; cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost);
    const double kk = KIND == 0 ? 32 : 64, cpm = best / (4.0 * rounds);
    printf("%s N=%3d: %6.1f cycles/MMA  %7.0f flop/cycle/SM  timeout=%d\n", KIND == 0 ? "mxf8f6f4 K=32" : "mxf4     K=64", N,
           cpm, 2.0 * 128 * N * kk / cpm, e);
  }
}

int main() {
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* cyc; cudaMalloc(&cyc, sizeof(unsigned long long) * 2 * sms);
  int* err; cudaMalloc(&err, 4); cudaMemset(err, 0, 4);
  run<0>(sms, cyc, err);
  run<1>(sms, cyc, err);
  return 0;
}
