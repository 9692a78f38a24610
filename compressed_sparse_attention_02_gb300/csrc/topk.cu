// Exact top-k of the lightning-indexer scores.  Page "CSA / HCA" (zdszero,
// hca_csa), "CSA：轻压缩 + 稀疏选择" (Top-k over I_{t,:}, all visible entries
// compete, window included); indices reported in ascending entry order
// ("DeepSeek 注意力结构对比" CSA2 section: sorted by position); equal scores
// are broken toward the smaller entry index.
//
// Scores become order-preserving 32-bit keys (sign-magnitude flip; -0 is
// folded into +0 and NaN maps to the smallest key).  One 512-thread CTA finds
// the k-th largest key of up to 16384 items held in shared memory with four
// 8-bit radix passes (shared-memory histograms, one block scan per pass to
// locate the digit), then compacts, in position order, every key above the
// threshold plus the first ties at it: positions ascend, so the output is
// already sorted.  Long rows are split into chunks whose local top-k (an exact
// superset of the global one) feed a second, merging selection.
#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t score_key(float f) {
  f = f + 0.0f;  // -0 -> +0
  if (f != f) return 0u;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

struct SelectSmem {
  int hist[256];
  int wsum[kWarps];
  int bucket;
  int above;
};

// Exclusive block-wide prefix sum of v; *total receives the sum over the block.
__device__ int block_excl_scan(int v, SelectSmem& sm, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sm.wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? sm.wsum[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < kWarps) sm.wsum[lane] = w;
  }
  __syncthreads();
  const int before = warp > 0 ? sm.wsum[warp - 1] : 0;
  *total = sm.wsum[kWarps - 1];
  __syncthreads();
  return before + x - v;
}

// Selects the kk largest of keys[0..n) (kk <= n), ties toward the smaller
// position, and calls emit(position, slot) for each with slots 0..kk-1 in
// ascending position order.
template <class Emit>
__device__ void block_select(const uint32_t* keys, int n, int kk, SelectSmem& sm, Emit emit) {
  const int tid = threadIdx.x;
  uint32_t thr = 0u;
  int ties = n;  // take everything when kk == n
  if (kk < n) {
    uint32_t prefix = 0u, mask = 0u;
    int remaining = kk;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kThreads) sm.hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < n; i += kThreads) {
        const uint32_t key = keys[i];
        if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 0xFFu], 1);
      }
      __syncthreads();
      // Bins from the top digit down: thread j holds bin 255-j.
      const int c = tid < 256 ? sm.hist[255 - tid] : 0;
      int tot;
      const int excl = block_excl_scan(c, sm, &tot);
      if (tid < 256 && excl < remaining && excl + c >= remaining) {
        sm.bucket = 255 - tid;
        sm.above = excl;
      }
      __syncthreads();
      remaining -= sm.above;
      prefix |= static_cast<uint32_t>(sm.bucket) << shift;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    thr = prefix;
    ties = remaining;
  }
  // Compaction in position order: each thread owns a contiguous segment.
  const int per = (n + kThreads - 1) / kThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int gt = 0, eq = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[i];
    gt += key > thr;
    eq += key == thr;
  }
  int tot;
  const int eq_before = block_excl_scan(eq, sm, &tot);
  const int take = max(0, min(eq, ties - eq_before));
  int slot = block_excl_scan(gt + take, sm, &tot);
  int seen = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[i];
    if (key > thr) {
      emit(i, slot++);
    } else if (key == thr) {
      if (seen < take) emit(i, slot++);
      ++seen;
    }
  }
}

__device__ __forceinline__ int64_t visible_entries(const TopkArgs& a, int b, int q) {
  const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[static_cast<int64_t>(b) * a.Q + q]) : a.pos_base + q;
  int64_t V = t >= 0 ? (t + 1) / a.m : 0;
  return V > a.n_cap ? a.n_cap : V;
}

// Pass 1: top-k of one chunk of one (sequence, query) row.  With a single
// chunk the result is final; otherwise it is a candidate list.
__global__ void __launch_bounds__(kThreads) topk_chunk_kernel(const TopkArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ SelectSmem sm;
  const int b = blockIdx.z, q = blockIdx.y, c = blockIdx.x;
  const int64_t row = static_cast<int64_t>(b) * a.Q + q;
  const int64_t V = visible_entries(a, b, q);
  const int64_t c0 = static_cast<int64_t>(c) * a.chunk;
  const int n = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(a.chunk), V - c0)));
  const int kk = min(a.k, n);
  const bool final_pass = a.n_chunks == 1;

  const float* src = a.scores + row * a.score_ld + c0;
  for (int i = threadIdx.x; i < n; i += kThreads) keys[i] = score_key(src[i]);
  __syncthreads();

  if (final_pass) {
    int32_t* idx = a.idx_out + row * a.k;
    float* sc = a.score_out ? a.score_out + row * a.k : nullptr;
    block_select(keys, n, kk, sm, [&](int pos, int slot) {
      idx[slot] = static_cast<int32_t>(c0 + pos);
      if (sc) sc[slot] = key_score(keys[pos]);
    });
    for (int j = kk + threadIdx.x; j < a.k; j += kThreads) {
      idx[j] = -1;
      if (sc) sc[j] = -INFINITY;
    }
  } else {
    if (n <= 0) return;
    uint32_t* ck = a.cand_key + (row * a.n_chunks + c) * a.k;
    int32_t* ci = a.cand_idx + (row * a.n_chunks + c) * a.k;
    block_select(keys, n, kk, sm, [&](int pos, int slot) {
      ck[slot] = keys[pos];
      ci[slot] = static_cast<int32_t>(c0 + pos);
    });
  }
}

// Pass 2: merge the per-chunk candidates of one row (already in ascending
// entry order chunk after chunk) into the final top-k.
__global__ void __launch_bounds__(kThreads) topk_merge_kernel(const TopkArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ SelectSmem sm;
  const int b = blockIdx.y, q = blockIdx.x;
  const int64_t row = static_cast<int64_t>(b) * a.Q + q;
  const int64_t V = visible_entries(a, b, q);
  int32_t* pos_idx = reinterpret_cast<int32_t*>(keys + kTopkMaxItems);

  int total = 0;
  for (int c = 0; c < a.n_chunks; ++c) {
    const int64_t nc = max(static_cast<int64_t>(0), min(static_cast<int64_t>(a.chunk), V - static_cast<int64_t>(c) * a.chunk));
    const int cnt = static_cast<int>(min(static_cast<int64_t>(a.k), nc));
    const uint32_t* ck = a.cand_key + (row * a.n_chunks + c) * a.k;
    const int32_t* ci = a.cand_idx + (row * a.n_chunks + c) * a.k;
    for (int j = threadIdx.x; j < cnt; j += kThreads) {
      keys[total + j] = ck[j];
      pos_idx[total + j] = ci[j];
    }
    total += cnt;
  }
  __syncthreads();
  const int kk = min(a.k, total);
  int32_t* idx = a.idx_out + row * a.k;
  float* sc = a.score_out ? a.score_out + row * a.k : nullptr;
  block_select(keys, total, kk, sm, [&](int pos, int slot) {
    idx[slot] = pos_idx[pos];
    if (sc) sc[slot] = key_score(keys[pos]);
  });
  for (int j = kk + threadIdx.x; j < a.k; j += kThreads) {
    idx[j] = -1;
    if (sc) sc[j] = -INFINITY;
  }
}

}  // namespace

void topk_chunking(int64_t rows, int64_t n_cap, int k, int* chunk, int* n_chunks) {
  // Start from the largest chunk one block holds; halve it while the first
  // pass would leave most SMs idle, as long as chunks stay well above k and
  // the merge still fits one block.
  int64_t ch = kTopkMaxItems;
  auto count = [&](int64_t c) { return (n_cap + c - 1) / c; };
  while (ch / 2 >= 2LL * k && ch / 2 >= 1024 && rows * count(ch) < 2 * 152 &&
         count(ch / 2) * k <= kTopkMaxItems)
    ch /= 2;
  int64_t nc = count(ch);
  if (nc < 1) nc = 1;
  *chunk = static_cast<int>(ch);
  *n_chunks = static_cast<int>(nc);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.B <= 0 || a.Q <= 0) return cudaSuccess;
  const size_t smem1 = static_cast<size_t>(a.chunk) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem1));
  if (e != cudaSuccess) return e;
  topk_chunk_kernel<<<dim3(a.n_chunks, a.Q, a.B), kThreads, smem1, stream>>>(a);
  if ((e = counted(cudaGetLastError())) != cudaSuccess) return e;
  if (a.n_chunks > 1) {
    const size_t smem2 = static_cast<size_t>(kTopkMaxItems) * 8;
    e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem2));
    if (e != cudaSuccess) return e;
    topk_merge_kernel<<<dim3(a.Q, a.B), kThreads, smem2, stream>>>(a);
    e = counted(cudaGetLastError());
  }
  return e;
}

}  // namespace csa
