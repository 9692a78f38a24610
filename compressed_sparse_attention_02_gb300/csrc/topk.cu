// Exact top-k of the lightning-indexer scores.  Page "CSA / HCA" (zdszero,
// hca_csa), "CSA：轻压缩 + 稀疏选择" (Top-k over I_{t,:}, all visible entries
// compete, window included); indices reported in ascending entry order
// ("DeepSeek 注意力结构对比" CSA2 section: sorted by position); equal scores
// are broken toward the smaller entry index.
//
// Scores become order-preserving 32-bit keys (sign-magnitude flip; -0 is
// folded into +0 and NaN maps to the smallest key).  One 1024-thread CTA
// holds up to 32768 keys of a row in shared memory and finds the k-th largest
// by successive refinement: the current key interval [lo, hi] is cut into
// 2048 equal bins (the keys spread over many bins, so the shared-memory
// histogram sees few conflicting atomics), the bin holding the k-th key
// becomes the next interval, and the search stops when that bin holds exactly
// the keys still needed or a single key value (at most four passes for 32-bit
// keys).  A compaction in position order (warp ballots, one scan over warps)
// then emits every key above the threshold plus the first ties at it, so the
// output is already sorted by entry.  Rows longer than 32768 are cut into
// chunks whose local top-k (an exact superset of the global one) are merged
// by a second selection.
#include "keys.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kChunk = 32768;  // keys one CTA selects from

constexpr int kCandCap = 4096;  // keys of the crossing digit resolved in shared memory

struct SelectSmem {
  int hist[kBins];
  int wval[kWarps];
  int wtotal;
  uint32_t wmin[kWarps], wmax[kWarps];
  int bin, above, in_bin;
  int n_cand;
  uint32_t cand[kCandCap];
};

// Exclusive scan over the 32 warps of one value per warp (every lane of a
// warp passes the same `v`); returns the warp's prefix, *total the sum.
__device__ int warp_values_scan(int v, SelectSmem& sm, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sm.wval[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int x = sm.wval[lane];
    int incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    sm.wval[lane] = incl - x;
    if (lane == 31) sm.wtotal = incl;
  }
  __syncthreads();
  const int r = sm.wval[warp];
  *total = sm.wtotal;
  __syncthreads();
  return r;
}

// Emits, in position order, every key > thr and the first `ties` keys == thr.
// Warp w owns positions [w*span, (w+1)*span); its lanes visit them 32 at a
// time; one scan over warps gives each warp its first output slot.
template <class Emit>
__device__ void compact_in_order(const uint32_t* keys, int n, uint32_t thr, int ties, SelectSmem& sm, Emit emit) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int span = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int p0 = min(n, warp * span), p1 = min(n, p0 + span);
  int gt = 0, eq = 0;
  for (int p = p0 + lane; p < p1; p += 32) {
    const uint32_t k = keys[p];
    gt += k > thr;
    eq += k == thr;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, off);
    eq += __shfl_xor_sync(0xffffffffu, eq, off);
  }
  int total;
  const int eq_before = warp_values_scan(eq, sm, &total);
  const int take = max(0, min(eq, ties - eq_before));
  int slot = warp_values_scan(gt + take, sm, &total);
  int seen = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    const uint32_t k = p < p1 ? keys[p] : 0u;
    const bool is_gt = p < p1 && k > thr;
    const bool is_eq = p < p1 && k == thr;
    const unsigned eqm = __ballot_sync(0xffffffffu, is_eq);
    const bool take_it = is_gt || (is_eq && seen + __popc(eqm & lt) < take);
    const unsigned selm = __ballot_sync(0xffffffffu, take_it);
    if (take_it) emit(p, slot + __popc(selm & lt));
    slot += __popc(selm);
    seen += __popc(eqm);
  }
}

// Finds, among the counts hist[0..nb) scanned from the top bin down, the bin
// where the running count first reaches `need`; sets sm.bin, sm.above (count
// in higher bins) and sm.in_bin.  Every thread holds nb / kThreads bins.
__device__ void find_crossing(const int* hist_s, const uint32_t* hist_g, int nb, int need, SelectSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int per = nb / kThreads;  // 1 or 2
  const int b0 = nb - 1 - per * tid;
  int c[2] = {0, 0};
  for (int u = 0; u < per; ++u) c[u] = hist_g ? static_cast<int>(__ldg(hist_g + b0 - u)) : hist_s[b0 - u];
  const int x = c[0] + c[1];
  int incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  int total;
  const int wprefix = warp_values_scan(__shfl_sync(0xffffffffu, incl, 31), sm, &total);
  int cum = wprefix + incl - x;
  for (int u = 0; u < per; ++u) {
    if (cum < need && cum + c[u] >= need) {
      sm.bin = b0 - u;
      sm.above = cum;
      sm.in_bin = c[u];
    }
    cum += c[u];
  }
  __syncthreads();
}

// Selects the kk largest of keys[0..n) (kk <= n <= kChunk), ties toward the
// smaller position, and calls emit(position, slot) for each, with slots
// 0..kk-1 in ascending position order.  Warp w owns positions
// [w*span, (w+1)*span); its lanes visit them 32 at a time.
template <class Emit>
__device__ void block_select(const uint32_t* keys, int n, int kk, SelectSmem& sm, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int span = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int p0 = min(n, warp * span), p1 = min(n, p0 + span);

  uint32_t thr = 0u;
  int ties = n;  // kk == n: everything is taken
  if (kk < n) {
    // key interval of the row
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    for (int p = p0 + lane; p < p1; p += 32) {
      const uint32_t k = keys[p];
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
    }
    if (lane == 0) {
      sm.wmin[warp] = kmin;
      sm.wmax[warp] = kmax;
    }
    __syncthreads();
    uint32_t lo = sm.wmin[0], hi = sm.wmax[0];
    for (int w = 1; w < kWarps; ++w) {
      lo = min(lo, sm.wmin[w]);
      hi = max(hi, sm.wmax[w]);
    }
    int remaining = kk;
    bool whole = false;
    while (lo < hi) {
      const uint64_t R = static_cast<uint64_t>(hi - lo) + 1u;
      for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = 0;
      __syncthreads();
      for (int p = p0 + lane; p < p1; p += 32) {
        const uint32_t k = keys[p];
        if (k >= lo && k <= hi)
          atomicAdd(&sm.hist[static_cast<int>(static_cast<uint64_t>(k - lo) * kBins / R)], 1);
      }
      __syncthreads();
      // Thread t owns bins 2047-2t and 2046-2t: counts from the top bin down.
      const int b0 = kBins - 1 - 2 * tid;
      const int c0 = sm.hist[b0], c1 = sm.hist[b0 - 1];
      const int x = c0 + c1;
      int incl = x;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      int total;
      const int wprefix = warp_values_scan(__shfl_sync(0xffffffffu, incl, 31), sm, &total);
      const int excl = wprefix + incl - x;  // keys in the bins above this thread's two
      if (excl < remaining && excl + c0 >= remaining) {
        sm.bin = b0;
        sm.above = excl;
        sm.in_bin = c0;
      } else if (excl + c0 < remaining && excl + x >= remaining) {
        sm.bin = b0 - 1;
        sm.above = excl + c0;
        sm.in_bin = c1;
      }
      __syncthreads();
      const int bin = sm.bin;
      remaining -= sm.above;
      const bool exact_bin = sm.in_bin == remaining;
      __syncthreads();
      // keys of bin b: lo + ceil(b*R/kBins) .. lo + ceil((b+1)*R/kBins) - 1
      const uint32_t blo = lo + static_cast<uint32_t>((static_cast<uint64_t>(bin) * R + kBins - 1) / kBins);
      const uint32_t bhi =
          lo + static_cast<uint32_t>((static_cast<uint64_t>(bin + 1) * R + kBins - 1) / kBins) - 1u;
      lo = blo;
      hi = bhi;
      if (exact_bin) {  // the whole bin is taken: select every key >= lo
        whole = true;
        break;
      }
    }
    thr = lo;
    ties = whole ? n : remaining;
  }

  compact_in_order(keys, n, thr, ties, sm, emit);
}

__device__ __forceinline__ int64_t visible_entries(const TopkArgs& a, int b, int q) {
  const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[static_cast<int64_t>(b) * a.Q + q]) : a.pos_base + q;
  int64_t V = t >= 0 ? (t + 1) / a.m : 0;
  return V > a.n_cap ? a.n_cap : V;
}

// Pass 1: top-k of one chunk of one (sequence, query) row.  With a single
// chunk the result is final; otherwise it is a candidate list.
__global__ void __launch_bounds__(kThreads, 1) topk_chunk_kernel(const TopkArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ SelectSmem sm;
  const int b = blockIdx.z, q = blockIdx.y, c = blockIdx.x;
  const int64_t row = static_cast<int64_t>(b) * a.Q + q;
  const int64_t V = visible_entries(a, b, q);
  const int64_t c0 = static_cast<int64_t>(c) * a.chunk;
  const int n = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(a.chunk), V - c0)));
  const int kk = min(a.k, n);
  const bool final_pass = a.n_chunks == 1;
  if (!final_pass && n <= 0) return;

  const float* src = a.scores + row * a.score_ld + c0;
  if (final_pass && a.hist && kk < n) {
    // The indexer counted the row's first digits: go straight to the digit
    // holding the k-th key and resolve only that digit's keys.
    find_crossing(nullptr, a.hist + row * kKeyBins, kKeyBins, kk, sm);
    const uint32_t dstar = static_cast<uint32_t>(sm.bin);
    const int remaining = kk - sm.above;
    const bool whole = sm.in_bin == remaining;
    if (threadIdx.x == 0) sm.n_cand = 0;
    // all loads first (independent, so they overlap), then the candidates
    for (int i = threadIdx.x; i < n; i += kThreads) keys[i] = score_key(__ldg(src + i));
    __syncthreads();
    const int lane = threadIdx.x & 31;
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + threadIdx.x;
      const uint32_t key = i < n ? keys[i] : 0u;
      const bool c = !whole && i < n && (key >> kKeyBinShift) == dstar;
      const unsigned m = __ballot_sync(0xffffffffu, c);
      int pos0 = 0;
      if (m && lane == 0) pos0 = atomicAdd(&sm.n_cand, __popc(m));
      pos0 = __shfl_sync(0xffffffffu, pos0, 0);
      const int pos = pos0 + __popc(m & ((1u << lane) - 1u));
      if (c && pos < kCandCap) sm.cand[pos] = key;
    }
    __syncthreads();
    uint32_t thr;
    int ties;
    if (whole) {
      thr = dstar << kKeyBinShift;  // every key of the digit is taken
      ties = n;
    } else if (sm.n_cand <= kCandCap) {
      // two more digits (11 + 10 bits) over the candidates only
      const int nc = sm.n_cand;
      uint32_t prefix = dstar << kKeyBinShift;
      int need = remaining;
      for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const int nb = pass == 0 ? 2048 : 1024;
        const uint32_t mask = pass == 0 ? 0xFFE00000u : 0xFFFFFC00u;
        for (int i = threadIdx.x; i < nb; i += kThreads) sm.hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < nc; i += kThreads) {
          const uint32_t k = sm.cand[i];
          if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & (nb - 1)], 1);
        }
        __syncthreads();
        find_crossing(sm.hist, nullptr, nb, need, sm);
        prefix |= static_cast<uint32_t>(sm.bin) << shift;
        need -= sm.above;
        __syncthreads();
      }
      thr = prefix;
      ties = need;
    } else {
      // pathological digit (more than kCandCap equal-digit keys): refine
      // over the whole row instead
      block_select(keys, n, kk, sm, [&](int pos, int slot) {
        a.idx_out[row * a.k + slot] = static_cast<int32_t>(c0 + pos);
        if (a.score_out) a.score_out[row * a.k + slot] = key_score(keys[pos]);
      });
      for (int j = kk + threadIdx.x; j < a.k; j += kThreads) {
        a.idx_out[row * a.k + j] = -1;
        if (a.score_out) a.score_out[row * a.k + j] = -INFINITY;
      }
      return;
    }
    int32_t* idx = a.idx_out + row * a.k;
    float* sc = a.score_out ? a.score_out + row * a.k : nullptr;
    compact_in_order(keys, n, thr, ties, sm, [&](int pos, int slot) {
      idx[slot] = static_cast<int32_t>(c0 + pos);
      if (sc) sc[slot] = key_score(keys[pos]);
    });
    for (int j = kk + threadIdx.x; j < a.k; j += kThreads) {
      idx[j] = -1;
      if (sc) sc[j] = -INFINITY;
    }
    return;
  }
  for (int i = threadIdx.x; i < n; i += kThreads) keys[i] = score_key(__ldg(src + i));
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
    uint32_t* ck = a.cand_key + (row * a.n_chunks + c) * a.k;
    int32_t* ci = a.cand_idx + (row * a.n_chunks + c) * a.k;
    block_select(keys, n, kk, sm, [&](int pos, int slot) {
      ck[slot] = keys[pos];
      ci[slot] = static_cast<int32_t>(c0 + pos);
    });
  }
}

// Pass 2: merge the per-chunk candidates of one row into the final top-k.
// Every chunk but the last non-empty one holds exactly k candidates (chunks
// are at least 2k long), so the candidates sit contiguously in chunk order,
// i.e. in ascending entry order.
__global__ void __launch_bounds__(kThreads, 1) topk_merge_kernel(const TopkArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ SelectSmem sm;
  const int b = blockIdx.y, q = blockIdx.x;
  const int64_t row = static_cast<int64_t>(b) * a.Q + q;
  const int64_t V = visible_entries(a, b, q);
  int32_t* pos_idx = reinterpret_cast<int32_t*>(keys + kTopkMaxItems);

  const int64_t n_full = V / a.chunk;
  const int64_t rest = V - n_full * a.chunk;
  const int total = static_cast<int>(n_full * a.k + min(static_cast<int64_t>(a.k), rest));
  const uint32_t* ck = a.cand_key + row * a.n_chunks * a.k;
  const int32_t* ci = a.cand_idx + row * a.n_chunks * a.k;
  for (int f = threadIdx.x; f < total; f += kThreads) {
    keys[f] = __ldg(ck + f);
    pos_idx[f] = __ldg(ci + f);
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
  (void)rows;
  (void)k;
  int64_t nc = (n_cap + kChunk - 1) / kChunk;
  if (nc < 1) nc = 1;
  *chunk = kChunk;
  *n_chunks = static_cast<int>(nc);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.B <= 0 || a.Q <= 0) return cudaSuccess;
  const int64_t items = a.n_chunks == 1 ? (a.n_cap < a.chunk ? a.n_cap : a.chunk) : a.chunk;
  const size_t smem1 = static_cast<size_t>(items) * 4;
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
