// Order-preserving 32-bit keys of fp32 scores and the first radix digit, shared by the indexer
// (which histograms the digit of every score it writes) and the top-k (which selects on the
// keys), so both sides derive the same digit from the same stored bits.
#pragma once
#include <cstdint>

namespace dsa {

// Larger score -> larger key; -0.0 and +0.0 map to the same key (they compare equal).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kHistBins = 2048;     // first radix digit: the top 11 bits of the key
constexpr int kHistShift = 21;
// The indexer histograms one key in kHistSample (positions s with s % kHistSample == 0): a
// sample from which the top-k picks a threshold bin, then counts exactly.
constexpr int kHistSample = 16;

__device__ __forceinline__ uint32_t first_digit(uint32_t key) { return key >> kHistShift; }

}  // namespace dsa
