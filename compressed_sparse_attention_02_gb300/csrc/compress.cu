// The compressor as a kernel of its own: one 64-thread CTA per (entry,
// sequence), 8 channels per thread (the entry routine is in compress.cuh).
// Decode calls run the same routine inside the top-k launch instead.
//
// The indexer's key compressor (index_key_entry in compress.cuh) runs in a
// kernel of its own (one warp per entry), or inside the compressor launch:
// with key arguments, warp 0 of each CTA also writes the indexer key of the
// CTA's entry after the main entry.
#include "compress.cuh"

namespace csa {
namespace {

constexpr int kThreads = kDim / 8;  // 64

template <int M>
__global__ void __launch_bounds__(kThreads) compress_kernel(const CompressArgs a, const CompressArgs k) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[kThreads / 32 + 1];
  compress_entry<M, 8>(a, blockIdx.y, blockIdx.x, threadIdx.x, red, [] { __syncthreads(); });
  if (k.B > 0 && threadIdx.x < 32) index_key_entry<M>(k, blockIdx.y, blockIdx.x, threadIdx.x, red + kThreads / 32);
}

// Bulk mode: the entry's source rows are four runs of M contiguous rows
// (block i of Z^a and C^a, block i-1 of Z^b and C^b), so one thread moves
// them into shared memory with four bulk copies on one barrier and the
// entry's threads read them from there: a CTA holds no row in registers, so
// more CTAs (and their copies) are resident per SM.
template <int M>
__global__ void __launch_bounds__(kThreads) compress_bulk_kernel(const CompressArgs a, const CompressArgs k) {
  __shared__ alignas(128) uint16_t stage[4 * M * kDim];
  __shared__ uint64_t bar;
  __shared__ float red[kThreads / 32 + 1];
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
  if (k.B > 0 && threadIdx.x < 32) index_key_entry<M>(k, b, e, threadIdx.x, red + kThreads / 32);
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
  index_key_entry<M>(a, blockIdx.y, e, lane, red + warp);
}

}  // namespace

void fill_rope_turns(double theta, uint64_t (&table)[kRope / 2]) {
  const double inv_two_pi = 0.15915494309189533576888376337251;
  for (int j = 0; j < kRope / 2; ++j)
    table[j] = static_cast<uint64_t>(ldexp(pow(theta, -2.0 * j / static_cast<double>(kRope)) * inv_two_pi, 64));
}

void fill_rope(CompressArgs* a) { fill_rope_turns(a->rope_theta, a->rope_turns); }

cudaError_t launch_compress(const CompressArgs& args, cudaStream_t stream, const CompressArgs* keys) {
  if (args.B <= 0) return cudaSuccess;
  CompressArgs a = args;
  fill_rope(&a);
  CompressArgs k = {};  // B = 0: no indexer keys
  if (keys) {
    if (keys->mode != 0 || args.mode != 0 || keys->B != args.B || keys->m != args.m || keys->n_new != args.n_new ||
        keys->entry0 != args.entry0)
      return cudaErrorInvalidValue;
    k = *keys;
    fill_rope(&k);
  }
  dim3 grid(a.mode == 0 ? static_cast<unsigned>(a.n_new) : 1u, static_cast<unsigned>(a.B));
  if (grid.x == 0) return cudaSuccess;
  // Staged rows from about one wave of CTAs on: below that the launch is
  // latency-bound and the register form, which issues its loads at once,
  // is a little faster (prefill chunks of 4096 tokens: 13.0 against 14.5 us).
  constexpr int64_t kStagedMinEntries = 2048;
  if (a.mode == 0 && static_cast<int64_t>(a.n_new) * a.B >= kStagedMinEntries) switch (a.m) {
      case 1: return launch_pdl(compress_bulk_kernel<1>, grid, dim3(kThreads), 0, stream, a, k);
      case 2: return launch_pdl(compress_bulk_kernel<2>, grid, dim3(kThreads), 0, stream, a, k);
      case 4: return launch_pdl(compress_bulk_kernel<4>, grid, dim3(kThreads), 0, stream, a, k);
      case 8: return launch_pdl(compress_bulk_kernel<8>, grid, dim3(kThreads), 0, stream, a, k);
      default: return cudaErrorInvalidValue;
    }
  switch (a.m) {
    case 1: return launch_pdl(compress_kernel<1>, grid, dim3(kThreads), 0, stream, a, k);
    case 2: return launch_pdl(compress_kernel<2>, grid, dim3(kThreads), 0, stream, a, k);
    case 4: return launch_pdl(compress_kernel<4>, grid, dim3(kThreads), 0, stream, a, k);
    case 8: return launch_pdl(compress_kernel<8>, grid, dim3(kThreads), 0, stream, a, k);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa

namespace csa {

cudaError_t launch_index_keys(const CompressArgs& args, cudaStream_t stream) {
  if (args.B <= 0 || args.n_new <= 0) return cudaSuccess;
  if (args.mode != 0) return cudaErrorInvalidValue;
  CompressArgs a = args;
  fill_rope(&a);
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
