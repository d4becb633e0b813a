// Device helpers shared by the layer's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Device error word bits (read back by moe_sync / the next call).
enum : int32_t { kErrExpertRange = 1, kErrTimeout = 2, kErrShape = 4 };

__device__ __forceinline__ void raise_error(int32_t* err, int32_t bit) {
  atomicOr(err, bit);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
  return __uint_as_float(b << 16);
}

// The block exponent of the dynamic FP8 scheme, from a non-negative fp32 amax:
// the smallest integer e with amax <= 448 * 2^e, limited to [-127, 127];
// amax = 0 gives 0.  With amax = 1.f * 2^E (normal) and 448 = 1.75 * 2^8 the
// answer is E - 8 when the significand 1.f is at most 1.75, else E - 7.  A
// subnormal amax is below 448 * 2^-127, so e = -127.
__device__ __forceinline__ int fp8_block_exponent(float amax) {
  const uint32_t u = __float_as_uint(amax);
  if (u == 0u) return 0;
  const int ebits = (int)(u >> 23);
  if (ebits == 0) return -127;
  const int E = ebits - 127;
  const uint32_t frac = u & 0x7FFFFFu;
  int e = (frac <= 0x600000u) ? E - 8 : E - 7;  // 0x600000 = significand 1.75
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^k as fp32 for k in [-126, 127].
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// Two fp32 values -> packed E4M3 pair (lo = first byte), nearest-even,
// saturating to +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Scales v by 2^-e exactly (e in [-127, 127]) before E4M3 rounding.  Done in
// two power-of-two steps so that neither factor leaves the fp32 normal range.
__device__ __forceinline__ float scale_pow2_neg(float v, int e) {
  const int a = -e / 2, b = -e - a;
  return v * exp2i(a) * exp2i(b);
}

// Four E2M1 codes packed in the low 16 bits of `codes` (element 0 in the low
// nibble) -> two f16x2 words, element order preserved.
__device__ __forceinline__ void e2m1x4_to_f16x4(uint32_t codes, uint32_t& h01, uint32_t& h23) {
  asm("{\n\t.reg .b8 b0, b1;\n\t"
      "mov.b16 {b0, b1}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t}"
      : "=r"(h01), "=r"(h23)
      : "h"((uint16_t)(codes & 0xFFFFu)));
}

// Two E4M3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// acc += a.lo * b.lo + a.hi * b.hi with f16 operands and fp32 accumulation
// (each f16 product is exact in fp32).
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

// Quantises 8 consecutive bf16 values; the four lanes of a quad (one 32-block)
// agree on the block exponent.  Returns the 8 codes; *e gets the exponent.
__device__ __forceinline__ uint2 quant8(const uint4 v, unsigned quad, int* e_out) {
  float f[8];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 2));
  const int e = fp8_block_exponent(amax);
  uint32_t c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    c[j] = e4m3x2(scale_pow2_neg(f[2 * j], e), scale_pow2_neg(f[2 * j + 1], e));
  *e_out = e;
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// FP4-activation variant: the smallest integer e with amax <= 6 * 2^e,
// limited to [-127, 127]; amax = 0 gives 0.  With amax = 1.f * 2^E (normal)
// and 6 = 1.5 * 2^2: E - 2 when the significand is at most 1.5, else E - 1.
// A subnormal amax is below 6 * 2^-127, so e = -127.
__device__ __forceinline__ int fp4_block_exponent(float amax) {
  const uint32_t u = __float_as_uint(amax);
  if (u == 0u) return 0;
  const int ebits = (int)(u >> 23);
  if (ebits == 0) return -127;
  const int E = ebits - 127;
  int e = ((u & 0x7FFFFFu) <= 0x400000u) ? E - 2 : E - 1;  // 0x400000 = significand 1.5
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Two fp32 values (already scaled into [-6, 6]) -> one byte of two E2M1
// codes, lo in the low nibble; nearest-even.  The sign bit of each code is
// taken from its input, so a negative value that rounds to zero gives -0.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "mov.b16 %0, {t, t};\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return ((uint32_t)r & 0x77u) | ((__float_as_uint(lo) >> 28) & 0x8u) | ((__float_as_uint(hi) >> 24) & 0x80u);
}

// Quantises 8 consecutive bf16 values to E2M1 (the FP4-activation variant);
// the four lanes of a quad (one 32-block) agree on the block exponent.
// Returns the 8 codes packed in 4 bytes (element 0 in the low nibble of byte
// 0); *e gets the exponent.
__device__ __forceinline__ uint32_t quant4(const uint4 v, unsigned quad, int* e_out) {
  float f[8];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 2));
  const int e = fp4_block_exponent(amax);
  uint32_t c = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) c |= e2m1x2(scale_pow2_neg(f[2 * j], e), scale_pow2_neg(f[2 * j + 1], e)) << (8 * j);
  *e_out = e;
  return c;
}

// *p += v at device scope with acquire-release order; returns the old value.
// Used by one thread after a CTA barrier: it publishes the writes the barrier
// ordered before it and, for the thread that sees the final count, acquires
// the writes every other CTA published the same way.
__device__ __forceinline__ int atomic_add_acq_rel(int32_t* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has finished and flushed its writes (a no-op when the kernel was not
// launched as a dependent), then let the next kernel start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

}  // namespace moe
