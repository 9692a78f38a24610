// The FP4 entry arithmetic shared by the quantizer and the compressor's
// FP4 store ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §16.1): a group of
// 16 values gets the E4M3 scale nearest to amax/6, each value the E2M1 code
// nearest to value/scale (saturating); both quotients in binary32.
#pragma once

#include <stdint.h>

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

namespace csa {

// The scale code of a group and its value (zero for an all-zero group).
__device__ __forceinline__ uint8_t fp4_scale_code(float amax, float* s) {
  const __nv_fp8_storage_t sc = __nv_cvt_float_to_fp8(__fdiv_rn(amax, 6.0f), __NV_SATFINITE, __NV_E4M3);
  *s = __half2float(__half(__nv_cvt_fp8_to_halfraw(sc, __NV_E4M3)));
  return static_cast<uint8_t>(sc);
}

// Two values' E2M1 codes, the first in the low nibble (zero codes for s = 0).
__device__ __forceinline__ uint32_t fp4_pair_code(float x0, float x1, float s) {
  if (s == 0.f) return 0u;
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp4x2(make_float2(__fdiv_rn(x0, s), __fdiv_rn(x1, s)), __NV_E2M1, cudaRoundNearest));
}

// E8M0 scale of a 32-value block of an FP4 indexer row (§16.2 of the same
// page): e is the smallest exponent in -127..127 with 6 * 2^e >= amax, read
// off amax's bits (amax = f * 2^E, f in [1, 2): e = E - 2 if f <= 1.5, else
// E - 1; below 2^-126 the smallest scale already fits).  Returns the byte
// e + 127 and sets *inv = 2^-e, so that x * inv is the exact quotient x / s.
__device__ __forceinline__ uint8_t e8m0_scale_code(float amax, float* inv) {
  const uint32_t b = __float_as_uint(amax);
  int e = -127;
  if (b >= 0x00800000u) {
    const int E = static_cast<int>(b >> 23) - 127;
    e = (b & 0x007FFFFFu) <= 0x00400000u ? E - 2 : E - 1;
    if (e < -127) e = -127;
  }
  *inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  return static_cast<uint8_t>(e + 127);
}

// Two already-scaled values' E2M1 codes, the first in the low nibble.
__device__ __forceinline__ uint32_t e2m1_pair_code(float y0, float y1) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(make_float2(y0, y1), __NV_E2M1, cudaRoundNearest));
}

}  // namespace csa
