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

}  // namespace csa
