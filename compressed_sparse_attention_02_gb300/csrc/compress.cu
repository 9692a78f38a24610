// The compressor as a kernel of its own: one 64-thread CTA per (entry,
// sequence), 8 channels per thread (the entry routine is in compress.cuh).
// Decode calls run the same routine inside the top-k launch instead.
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
  switch (a.m) {
    case 1: return launch_pdl(compress_kernel<1>, grid, dim3(kThreads), 0, stream, a);
    case 2: return launch_pdl(compress_kernel<2>, grid, dim3(kThreads), 0, stream, a);
    case 4: return launch_pdl(compress_kernel<4>, grid, dim3(kThreads), 0, stream, a);
    case 8: return launch_pdl(compress_kernel<8>, grid, dim3(kThreads), 0, stream, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa
