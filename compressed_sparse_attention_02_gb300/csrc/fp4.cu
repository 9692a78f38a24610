// FP4 cache entries and FP4 indexer rows.
// Main KV ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §16.1: a
// Main KV entry of 512 FP4 values with one 1-byte E4M3 scale per 16 values,
// 288 bytes).  Layout of an entry: bytes 0..255 the E2M1 codes (channel 2j
// in the low nibble of byte j), bytes 256..287 the E4M3 scales (scale g for
// channels 16g..16g+15).  A group's scale is the E4M3 code nearest to
// amax/6 and a channel's code the E2M1 code nearest to x/scale, saturating,
// both quotients in binary32.
//
// One warp per entry, one lane per 16-channel group: two 16-byte loads, the
// group maximum, the scale, eight paired conversions, one 8-byte store of
// codes and one scale byte.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "fp4.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kRowsPerCta = 8;

__global__ void __launch_bounds__(32 * kRowsPerCta) quantize_kv_fp4_kernel(const int64_t n_rows, const uint16_t* in,
                                                                          const int64_t in_stride, uint8_t* out,
                                                                          const int64_t out_stride) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
  const int g = threadIdx.x & 31;
  if (row >= n_rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(in + row * in_stride + 16 * g);
  const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  float x[16];
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    x[2 * j] = __uint_as_float(w[j] << 16);
    x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(x[2 * j]), fabsf(x[2 * j + 1])));
  }
  float s;
  const uint8_t sc = fp4_scale_code(amax, &s);
  uint32_t codes[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) codes[j >> 2] |= fp4_pair_code(x[2 * j], x[2 * j + 1], s) << (8 * (j & 3));
  uint8_t* dst = out + row * out_stride;
  *reinterpret_cast<uint2*>(dst + 8 * g) = make_uint2(codes[0], codes[1]);
  dst[kDim / 2 + g] = sc;
}

// FP4 indexer rows (§16.2: 128 E2M1 values, one E8M0 scale per 32): one warp
// per row, lane l takes channels 4l .. 4l+3 (block l/8); the block maximum
// over 8 lanes, the scale, two paired conversions, a 2-byte code store, and
// the scale byte into the row's place in its 512-byte atom.
constexpr int kIdxRowsPerCta = 8;

__global__ void __launch_bounds__(32 * kIdxRowsPerCta) quantize_index_fp4_kernel(const IndexFp4Rows a) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kIdxRowsPerCta + (threadIdx.x >> 5);
  if (w >= static_cast<int64_t>(a.B) * a.n_rows) return;
  const int lane = threadIdx.x & 31;
  const int64_t b = w / a.n_rows, j = w % a.n_rows, e = a.entry0 + j;
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(a.in + b * a.in_stride_b + j * kIdxDim) + lane);
  const float x[4] = {__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                      __uint_as_float(u.y & 0xFFFF0000u)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  float inv;
  const uint8_t sc = e8m0_scale_code(amax, &inv);
  const uint32_t c = e2m1_pair_code(x[0] * inv, x[1] * inv) | (e2m1_pair_code(x[2] * inv, x[3] * inv) << 8);
  *reinterpret_cast<uint16_t*>(a.codes + b * a.codes_stride_b + e * (kIdxDim / 2) + 2 * lane) =
      static_cast<uint16_t>(c);
  uint8_t* atom = a.sf + b * a.sf_stride_b + (e >> 7) * 512;
  if ((lane & 7) == 0) atom[16 * (e & 31) + 4 * ((e & 127) >> 5) + (lane >> 3)] = sc;
  if (a.zero_pad && lane == 0 && e < 32) *reinterpret_cast<uint2*>(atom + 16 * e + 8) = make_uint2(0u, 0u);
}

}  // namespace

cudaError_t launch_quantize_index_fp4(const IndexFp4Rows& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.n_rows;
  if (rows <= 0) return cudaSuccess;
  const int64_t ctas = (rows + kIdxRowsPerCta - 1) / kIdxRowsPerCta;
  if (ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
  return launch_pdl(quantize_index_fp4_kernel, dim3(static_cast<unsigned>(ctas)), dim3(32 * kIdxRowsPerCta), 0,
                    stream, a);
}

cudaError_t launch_quantize_kv_fp4(int64_t n_rows, const uint16_t* in, int64_t in_stride, uint8_t* out,
                                   int64_t out_stride, cudaStream_t stream) {
  if (n_rows <= 0) return cudaSuccess;
  const int64_t ctas = (n_rows + kRowsPerCta - 1) / kRowsPerCta;
  if (ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
  return launch_pdl(quantize_kv_fp4_kernel, dim3(static_cast<unsigned>(ctas)), dim3(32 * kRowsPerCta), 0, stream,
                    n_rows, in, in_stride, out, out_stride);
}

}  // namespace csa
