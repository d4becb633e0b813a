// GPU filler for synthetic MXFP4 expert banks.
//
// Same counter-based definition as synth/__init__.py: word j of a stream is
// mix64(key + (j + 1) * GAMMA) (SplitMix64 output function, Steele, Lea and
// Flood, OOPSLA 2014); byte i of the stream is byte (i mod 8), little-endian,
// of word i / 8.  Scale streams map each byte b to 127 + lo + (b mod (hi-lo+1)).
// The key of expert e's stream is fold(fold(fold(fold(0, seed), layer),
// 2*matrix + kind), e) with fold(k, v) = mix64(k + (v + 1) * GAMMA).
//
// This file holds no arithmetic of the MoE layer: it only produces input bytes.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t fold(uint64_t k, uint64_t v) { return mix64(k + (v + 1) * kGamma); }

__global__ void fill_kernel(uint8_t* base, uint64_t bytes_per_expert, int n_experts, int expert0,
                            uint64_t matrix_key, int is_scale, int lo, int n) {
  const uint64_t words_per_expert = (bytes_per_expert + 7) / 8;
  const uint64_t total = words_per_expert * (uint64_t)n_experts;
  for (uint64_t g = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t e = g / words_per_expert;
    const uint64_t j = g - e * words_per_expert;
    const uint64_t key = fold(matrix_key, (uint64_t)(expert0 + (int)e));
    uint64_t w = mix64(key + (j + 1) * kGamma);
    if (is_scale) {
      uint64_t out = 0;
      for (int b = 0; b < 8; ++b) {
        const uint32_t byte = (uint32_t)(w >> (8 * b)) & 0xFFu;
        out |= (uint64_t)((uint32_t)(127 + lo) + byte % (uint32_t)n) << (8 * b);
      }
      w = out;
    }
    uint8_t* dst = base + e * bytes_per_expert + j * 8;
    const uint64_t left = bytes_per_expert - j * 8;
    if (left >= 8 && ((uintptr_t)dst & 7) == 0) {
      *reinterpret_cast<uint64_t*>(dst) = w;
    } else {
      const int nb = left < 8 ? (int)left : 8;
      for (int b = 0; b < nb; ++b) dst[b] = (uint8_t)(w >> (8 * b));
    }
  }
}

}  // namespace

extern "C" {

// Fills n_experts consecutive expert streams (expert ids expert0 ..) of
// bytes_per_expert bytes each, starting at device pointer dst.
// kind 0 = packed E2M1 codes, kind 1 = UE8M0 scales with exponents in [lo, hi].
// Returns 0 on success, otherwise the cudaError_t of the launch.
int synth_fill(void* dst, unsigned long long bytes_per_expert, int n_experts, int expert0, int seed,
               int layer, int matrix, int kind, int lo, int hi, void* stream) {
  if (!dst || n_experts <= 0 || bytes_per_expert == 0) return (int)cudaErrorInvalidValue;
  uint64_t k = fold(0, (uint64_t)seed);
  k = fold(k, (uint64_t)layer);
  k = fold(k, (uint64_t)(2 * matrix + kind));
  const uint64_t words = (bytes_per_expert + 7) / 8 * (uint64_t)n_experts;
  uint64_t blocks = (words + 255) / 256;
  if (blocks > 152ull * 32) blocks = 152ull * 32;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      (uint8_t*)dst, bytes_per_expert, n_experts, expert0, k, kind, lo, hi - lo + 1);
  return (int)cudaGetLastError();
}

}  // extern "C"
