/* Host filler for synthetic byte streams: the same counter-based definition
 * as synth/__init__.py and synth/fill.cu (SplitMix64 output function of
 * key + (j + 1) * GAMMA for word j; byte i = byte i mod 8 of word i / 8).
 * Holds no arithmetic of the MoE layer. */
#include <stddef.h>
#include <stdint.h>

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* kind 0: raw bytes; kind 1: scale bytes 127 + lo + (b mod n). */
void synth_host_stream(uint8_t* dst, size_t n_bytes, uint64_t key, int kind, int lo, int n) {
  const uint64_t gamma = 0x9E3779B97F4A7C15ull;
  for (size_t i = 0; i < n_bytes; i += 8) {
    uint64_t w = mix64(key + (uint64_t)(i / 8 + 1) * gamma);
    for (size_t b = 0; b < 8 && i + b < n_bytes; ++b) {
      uint32_t v = (uint32_t)(w >> (8 * b)) & 0xFFu;
      dst[i + b] = kind ? (uint8_t)(127 + lo + (int)(v % (uint32_t)n)) : (uint8_t)v;
    }
  }
}
