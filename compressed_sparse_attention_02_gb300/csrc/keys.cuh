// Order-preserving 32-bit keys of fp32 scores, shared by the indexer (which
// histograms the keys' top bits while it scores) and the top-k selection.
#pragma once

#include <stdint.h>

namespace csa {

// Larger score -> larger key; -0 is folded into +0 and NaN maps to key 0
// (below every number).
__device__ __forceinline__ uint32_t score_key(float f) {
  f = f + 0.0f;
  if (f != f) return 0u;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// The first selection digit: the key's top 11 bits (sign, exponent, two
// mantissa bits), 2048 bins per row.
constexpr int kKeyBins = 2048;
constexpr int kKeyBinShift = 21;

}  // namespace csa
