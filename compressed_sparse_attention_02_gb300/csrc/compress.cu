// The compressor as a kernel of its own: one 64-thread CTA per (entry,
// sequence), 8 channels per thread (the entry routine is in compress.cuh).
// Decode calls run the same routine inside the top-k launch instead.
//
// The indexer's key compressor ([hca_csa] "CSA：轻压缩 + 稀疏选择": its own
// compressor at head_dim 128, then a Hadamard rotation so that the keys
// quantise well to FP8): the same steps at width 128, one warp per entry
// with 4 channels per lane, then H_128/sqrt(128) as butterflies (two stages
// in registers, five across lanes), then E4M3 with round-to-nearest-even
// and saturation at +-448.
#include <cuda_fp8.h>

#include "compress.cuh"

namespace csa {
namespace {

constexpr int kThreads = kDim / 8;  // 64

template <int M>
__global__ void __launch_bounds__(kThreads) compress_kernel(const CompressArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[kThreads / 32];
  compress_entry<M, 8>(a, blockIdx.y, blockIdx.x, threadIdx.x, red, [] { __syncthreads(); });
}

// Bulk mode: the entry's source rows are four runs of M contiguous rows
// (block i of Z^a and C^a, block i-1 of Z^b and C^b), so one thread moves
// them into shared memory with four bulk copies on one barrier and the
// entry's threads read them from there: a CTA holds no row in registers, so
// more CTAs (and their copies) are resident per SM.
template <int M>
__global__ void __launch_bounds__(kThreads) compress_bulk_kernel(const CompressArgs a) {
  __shared__ alignas(128) uint16_t stage[4 * M * kDim];
  __shared__ uint64_t bar;
  __shared__ float red[kThreads / 32];
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const int64_t e = blockIdx.x;
  const bool has_prev = a.entry0 + e > 0;
  constexpr uint32_t kRun = M * kDim * 2;  // bytes of M rows
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  if (threadIdx.x == 0) {
    const int64_t seq = static_cast<int64_t>(b) * M * a.n_new * kDim;
    mbar_arrive_expect_tx(&bar, (has_prev ? 4 : 2) * kRun);
    bulk_load(stage, a.Za + seq + M * e * kDim, kRun, &bar);
    bulk_load(stage + M * kDim, a.Ca + seq + M * e * kDim, kRun, &bar);
    if (has_prev) {  // block entry0-1 lives in the separate "previous block" rows
      const uint16_t* zb = e > 0 ? a.Zb + seq + M * (e - 1) * kDim : a.Zb_prev + static_cast<int64_t>(b) * M * kDim;
      const uint16_t* cb = e > 0 ? a.Cb + seq + M * (e - 1) * kDim : a.Cb_prev + static_cast<int64_t>(b) * M * kDim;
      bulk_load(stage + 2 * M * kDim, zb, kRun, &bar);
      bulk_load(stage + 3 * M * kDim, cb, kRun, &bar);
    }
  }
  if (!__syncthreads_and(mbar_wait(&bar, 0, a.status))) {
    mbar_wait(&bar, 0, a.status);  // no copy of ours stays in flight
    return;
  }
  const auto sync = [] { __syncthreads(); };
  compress_entry<M, 8, decltype(sync), true>(a, b, e, threadIdx.x, red, sync, stage);
}

constexpr int kKeyWarps = 4;  // entries per CTA of the key kernel

template <int M>
__global__ void __launch_bounds__(32 * kKeyWarps) index_key_kernel(const CompressArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[kKeyWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * kKeyWarps + warp;
  if (e >= a.n_new) return;  // warp-uniform
  float y[4];
  int64_t i;
  if (!compress_values<M, 4, kIdxDim>(a, blockIdx.y, e, lane, red + warp, [] { __syncwarp(); }, y, &i)) return;
  // H_128 x: butterflies (a, b) -> (a + b, a - b) over channel distance 1, 2
  // (within the lane's 4 channels), then 4 .. 64 (lanes 1 .. 16 apart)
  {
    const float s0 = y[0] + y[1], d0 = y[0] - y[1], s1 = y[2] + y[3], d1 = y[2] - y[3];
    y[0] = s0 + s1;
    y[1] = d0 + d1;
    y[2] = s0 - s1;
    y[3] = d0 - d1;
  }
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const bool upper = (lane >> st) & 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float o = __shfl_xor_sync(0xffffffffu, y[j], 1 << st);
      y[j] = upper ? o - y[j] : y[j] + o;
    }
  }
  constexpr float kInvSqrt128 = 0.088388347648318440550f;
  uint32_t codes = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    codes |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(y[j] * kInvSqrt128, __NV_SATFINITE, __NV_E4M3)) << (8 * j);
  *reinterpret_cast<uint32_t*>(a.key_out + static_cast<int64_t>(blockIdx.y) * a.kv_stride_b + i * kIdxDim +
                               4 * lane) = codes;
}

}  // namespace

void fill_inv_freq(CompressArgs* a) {
  for (int j = 0; j < kRope / 2; ++j) a->inv_freq[j] = pow(a->rope_theta, -2.0 * j / static_cast<double>(kRope));
}

cudaError_t launch_compress(const CompressArgs& args, cudaStream_t stream) {
  if (args.B <= 0) return cudaSuccess;
  CompressArgs a = args;
  fill_inv_freq(&a);
  dim3 grid(a.mode == 0 ? static_cast<unsigned>(a.n_new) : 1u, static_cast<unsigned>(a.B));
  if (grid.x == 0) return cudaSuccess;
  // Staged rows from about one wave of CTAs on: below that the launch is
  // latency-bound and the register form, which issues its loads at once,
  // is a little faster (prefill chunks of 4096 tokens: 13.0 against 14.5 us).
  constexpr int64_t kStagedMinEntries = 2048;
  if (a.mode == 0 && static_cast<int64_t>(a.n_new) * a.B >= kStagedMinEntries) switch (a.m) {
      case 1: return launch_pdl(compress_bulk_kernel<1>, grid, dim3(kThreads), 0, stream, a);
      case 2: return launch_pdl(compress_bulk_kernel<2>, grid, dim3(kThreads), 0, stream, a);
      case 4: return launch_pdl(compress_bulk_kernel<4>, grid, dim3(kThreads), 0, stream, a);
      case 8: return launch_pdl(compress_bulk_kernel<8>, grid, dim3(kThreads), 0, stream, a);
      default: return cudaErrorInvalidValue;
    }
  switch (a.m) {
    case 1: return launch_pdl(compress_kernel<1>, grid, dim3(kThreads), 0, stream, a);
    case 2: return launch_pdl(compress_kernel<2>, grid, dim3(kThreads), 0, stream, a);
    case 4: return launch_pdl(compress_kernel<4>, grid, dim3(kThreads), 0, stream, a);
    case 8: return launch_pdl(compress_kernel<8>, grid, dim3(kThreads), 0, stream, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa

namespace csa {

cudaError_t launch_index_keys(const CompressArgs& args, cudaStream_t stream) {
  if (args.B <= 0 || args.n_new <= 0) return cudaSuccess;
  if (args.mode != 0) return cudaErrorInvalidValue;
  CompressArgs a = args;
  fill_inv_freq(&a);
  const dim3 grid(static_cast<unsigned>((a.n_new + kKeyWarps - 1) / kKeyWarps), static_cast<unsigned>(a.B));
  const dim3 block(32 * kKeyWarps);
  switch (a.m) {
    case 1: return launch_pdl(index_key_kernel<1>, grid, block, 0, stream, a);
    case 2: return launch_pdl(index_key_kernel<2>, grid, block, 0, stream, a);
    case 4: return launch_pdl(index_key_kernel<4>, grid, block, 0, stream, a);
    case 8: return launch_pdl(index_key_kernel<8>, grid, block, 0, stream, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa
