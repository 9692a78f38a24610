// Exact top-k of the lightning-indexer scores.  Page "CSA / HCA" (zdszero,
// hca_csa), "CSA：轻压缩 + 稀疏选择" (Top-k over I_{t,:}, all visible entries
// compete, window included); indices reported in ascending entry order
// ("DeepSeek 注意力结构对比" CSA2 section: sorted by position); equal scores
// are broken toward the smaller entry index.
//
// Scores are compared as order-preserving 32-bit keys (keys.cuh).  While it
// scores, the indexer counts each row's keys by their top 11 bits (the
// "digit"), so the digit d* that holds the k-th largest key is known without
// another pass over the row.  One kernel then selects, one CTA per 4096 keys
// of a row:
//   filter  a key whose digit is above d* is selected.  Each thread reads 16
//           consecutive keys from shared memory and builds their half of a
//           32-bit word of the row's position bitmap.  A key whose digit is
//           d* is a candidate: the CTA gathers its candidates in shared
//           memory and appends them, with their positions, to the row's list
//           (one global atomic per CTA).
//   finish  the last CTA of the row to finish its filter (release/acquire on
//           a per-row counter; no CTA waits for another) loads the row's
//           bitmap and candidates together and resolves the candidates
//           exactly: the next 11 bits of their keys give the crossing bin;
//           when that bin holds at most 32 keys one warp ranks them by (key,
//           position), else a last 10-bit digit gives the threshold key and
//           the keys equal to it are taken in position order from a tie
//           bitmap.  The selected candidates are OR-ed into the bitmap, which
//           is then read out in position order (the ascending output), and
//           the selected scores are gathered last.
// When d* alone holds exactly the keys still needed, the filter selects all of
// d* and the finish only reads the bitmap out.  A row whose candidate list
// overflows is resolved from its scores in global memory (slower, exact).
//
// A decode step's compressor entry (compress.cuh) can ride along: one extra
// CTA per sequence computes it, so its latency hides behind the selection.
//
// The same kernel selects the hierarchical indexer's pool blocks (over the
// block scores, ceil(V/8) of them) and a Reindex layer's entries (over the
// pool's slots, mapped back to entries through the pool when written out);
// "DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §11.
#include "compress.cuh"
#include "keys.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 4096;     // keys per CTA: 16 consecutive keys per thread
constexpr int kLocalCap = 2048;  // candidates one CTA gathers before the row falls back
constexpr int kEmitWords = 8;    // bitmap words a thread reads per round of the read-out
constexpr int kBatch = 8;        // global loads a thread issues before using them (passes over global lists)
constexpr int kRoundWords = kThreads * kEmitWords;
static_assert(kItems == 16 * kThreads, "a thread covers half a bitmap word");
static_assert(kTopkCandCap == kRoundWords && kLocalCap == kTopkCandCap && kRoundWords >= kMaxTopk,
              "shared-memory reuse");

struct Crossing {
  int bin, above, in_bin;  // the bin, the count in higher bins, the count in it
};

struct __align__(16) Smem {
  union {
    struct {
      float vals[kItems];        // the CTA's scores
      uint32_t lkey[kLocalCap];  // its candidates
      int32_t lpos[kLocalCap];
    } f;
    struct {
      uint32_t ckey[kTopkCandCap];  // the row's candidates
      int32_t cpos[kTopkCandCap];
      uint32_t bm[kRoundWords];     // one read-out round of the row's position bitmap
      int32_t sel[kMaxTopk];        // the selected positions, ascending
    } c;
  } u;
  union {
    int hist[2048];           // digit counts
    int32_t xpos[kMaxTopk];   // extra selected positions (unordered)
  } h;
  int wsum[kWarps];
  int wval[kWarps];
  float red[kWarps];
  int wtotal;
  Crossing out;
  int n_local, last, nx, nsmall;
  unsigned cand_base;
  uint32_t small_key[32];  // the keys of a small crossing bin
  int32_t small_pos[32];
  uint64_t hist_bar, vals_bar;
};

// Exclusive scan over the warps of the block of one value per warp (every
// lane of a warp passes the same v); returns the warp's prefix, *total the sum.
__device__ int warps_scan(int v, Smem& sm, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sm.wval[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < kWarps ? sm.wval[lane] : 0;
    int incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane < kWarps) sm.wval[lane] = incl - x;
    if (lane == 31) sm.wtotal = incl;
  }
  __syncthreads();
  const int r = sm.wval[warp];
  *total = sm.wtotal;
  __syncthreads();
  return r;
}

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  return x;
}

// The block-wide exclusive prefix of this thread's count; *total the sum.
__device__ int block_prefix(int cnt, Smem& sm, int* total) {
  const int incl = warp_incl_scan(cnt);
  const int wbase = warps_scan(__shfl_sync(0xffffffffu, incl, 31), sm, total);
  return wbase + incl - cnt;
}

// Scanning the counts of nb (1024 or 2048) bins of sm.h.hist from the top bin
// down, finds the bin in which the running count first reaches `need`.  Thread
// t holds bins nb-1-per*t down to nb-per*(t+1); two barriers.  If the counts
// never reach `need` the result is {0, 0, 0}.
__device__ Crossing find_crossing(int nb, int need, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = nb / kThreads;  // 4 or 8
  const int lo = nb - per * (static_cast<int>(threadIdx.x) + 1);
  int c[8];
  const int4 v0 = *reinterpret_cast<const int4*>(sm.h.hist + lo + per - 4);
  const int4 v1 = per == 8 ? *reinterpret_cast<const int4*>(sm.h.hist + lo) : make_int4(0, 0, 0, 0);
  c[0] = v0.w, c[1] = v0.z, c[2] = v0.y, c[3] = v0.x;  // highest bin first
  c[4] = v1.w, c[5] = v1.z, c[6] = v1.y, c[7] = v1.x;
  int x = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) x += c[u];
  const int incl = warp_incl_scan(x);
  if (lane == 31) sm.wsum[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int s = sm.wsum[w];
    before += w < warp ? s : 0;
    total += s;
  }
  int cum = before + incl - x;
  if (cum < need && cum + x >= need) {
    const int top = lo + per - 1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < per && cum < need && cum + c[u] >= need) sm.out = Crossing{top - u, cum, c[u]};
      cum += c[u];
    }
  }
  __syncthreads();
  return total >= need ? sm.out : Crossing{0, 0, 0};
}

// Resolves the key digits below the first, 11 then 10 bits, among keys whose
// first digit is d*; key_at(i) for i < n gives the keys to count.  Returns the
// exact threshold key; *need becomes how many keys equal to it are taken and
// *n_eq how many there are.
template <class KeyAt>
__device__ uint32_t resolve_threshold(uint32_t dstar, int64_t n, KeyAt key_at, Smem& sm, int* need, int* n_eq) {
  uint32_t prefix = dstar << kKeyBinShift;
  int in_bin = 0;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    const int nb = pass == 0 ? 2048 : 1024;
    const uint32_t mask = pass == 0 ? 0xFFE00000u : 0xFFFFFC00u;
    for (int i = threadIdx.x; i < nb; i += kThreads) sm.h.hist[i] = 0;
    __syncthreads();
    for (int64_t i0 = 0; i0 < n; i0 += kBatch * kThreads) {  // kBatch independent loads in flight
      uint32_t kk[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int64_t i = i0 + u * kThreads + threadIdx.x;
        kk[u] = i < n ? key_at(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int64_t i = i0 + u * kThreads + threadIdx.x;
        if (i < n && (kk[u] & mask) == prefix) atomicAdd(&sm.h.hist[(kk[u] >> shift) & (nb - 1)], 1);
      }
    }
    __syncthreads();
    const Crossing c = find_crossing(nb, *need, sm);
    prefix |= static_cast<uint32_t>(c.bin) << shift;
    *need -= c.above;
    in_bin = c.in_bin;
  }
  *n_eq = in_bin;
  return prefix;
}

__device__ __forceinline__ void push_extra(Smem& sm, int32_t pos) {
  const int slot = atomicAdd(&sm.nx, 1);
  if (slot < kMaxTopk) sm.h.xpos[slot] = pos;
}

// Selects position pos: in the staged first round of the bitmap, or in the
// list of positions past it (rows longer than kRoundWords words).
__device__ __forceinline__ void mark(Smem& sm, int32_t pos) {
  if ((pos >> 5) < kRoundWords) atomicOr(&sm.u.c.bm[pos >> 5], 1u << (pos & 31));
  else push_extra(sm, pos);
}

// One bulk async copy global -> shared completing on `bar` (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// The number of keys of the row: its visible entries; or their blocks
// (vis_shift); or, with a pool, its valid slots: the pool holds
// nb = min(pool_blocks, ceil(V/8)) ascending blocks, all entries visible but
// those of block ceil(V/8)-1 past V, which can only be the pool's last.
// *ventries receives V.
// Score i of a row (fp32, or bf16 bits widened exactly).
__device__ __forceinline__ float row_score(const TopkArgs& a, int64_t row, int64_t i) {
  if (a.bf16_scores)
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(a.scores) +
                                                      row * a.score_ld + i))
                           << 16);
  return __ldg(a.scores + row * a.score_ld + i);
}

__device__ __forceinline__ int64_t row_extent(const TopkArgs& a, int b, int q, int64_t* ventries) {
  const int64_t row = static_cast<int64_t>(b) * a.Q + q;
  const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[row]) : a.pos_base + q;
  int64_t V = t >= 0 ? (t + 1) / a.m : 0;
  V = V > a.n_cap ? a.n_cap : V;
  *ventries = V;
  if (a.vis_shift) return (V + (int64_t(1) << a.vis_shift) - 1) >> a.vis_shift;
  if (a.pool) {
    const int64_t nvb = (V + kPoolBlock - 1) / kPoolBlock;
    const int64_t nb = nvb < a.pool_blocks ? nvb : a.pool_blocks;
    if (nb == 0) return 0;
    const int32_t last = __ldg(a.pool + row * a.pool_ld + nb - 1);
    return nb * kPoolBlock - (last == nvb - 1 ? nvb * kPoolBlock - V : 0);
  }
  return V;
}

// The entry a selected position stands for: itself, or with a pool the
// entry in the slot's block; -1 where that is no visible entry (only a pool
// that is not the Full layer's for this query leads there).
__device__ __forceinline__ int32_t out_entry(const TopkArgs& a, int64_t row, int64_t ventries, int32_t p) {
  if (!a.pool || p < 0) return p;
  const int32_t blk = __ldg(a.pool + row * a.pool_ld + (p / kPoolBlock));
  const int64_t e = static_cast<int64_t>(blk) * kPoolBlock + (p % kPoolBlock);
  return (blk < 0 || e >= ventries) ? -1 : static_cast<int32_t>(e);
}

// The `need` lowest positions of the tie bitmap go to the extra list.
__device__ void take_ties(const uint32_t* ties, int64_t nwords, int need, Smem& sm) {
  __syncthreads();  // the tie bits of every thread are in the bitmap
  int done = 0;
  for (int64_t w0 = 0; w0 < nwords && done < need; w0 += kThreads) {
    const int64_t w = w0 + threadIdx.x;
    uint32_t word = w < nwords ? __ldcg(ties + w) : 0u;
    int total;
    int before = done + block_prefix(__popc(word), sm, &total);
    while (word && before < need) {
      const int bit = __ffs(word) - 1;
      word &= word - 1;
      mark(sm, static_cast<int32_t>(w * 32 + bit));
      ++before;
    }
    done += total;
  }
}

// Calls f(key, position) for each of the row's nc candidates: from shared
// memory where the list is staged there, else from the global list, kBatch
// independent loads per thread at a time.  A position outside [0, V) (never
// written by this row's filter) reads as key 0 at position 0, the lowest key.
template <class F>
__device__ __forceinline__ void for_candidates(bool staged, int nc, const Smem& sm, const uint32_t* gkey,
                                               const int32_t* gpos, int64_t V, F f) {
  if (staged) {
    for (int i = threadIdx.x; i < nc; i += kThreads) f(sm.u.c.ckey[i], sm.u.c.cpos[i]);
    return;
  }
  for (int i0 = 0; i0 < nc; i0 += kBatch * kThreads) {
    uint32_t kk[kBatch];
    int32_t pp[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kThreads + static_cast<int>(threadIdx.x);
      kk[u] = i < nc ? __ldcg(gkey + i) : 0u;
      pp[u] = i < nc ? __ldcg(gpos + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kThreads + static_cast<int>(threadIdx.x);
      if (i >= nc) continue;
      const bool ok = pp[u] >= 0 && pp[u] < V;
      f(ok ? kk[u] : 0u, ok ? pp[u] : 0);
    }
  }
}

// Reads the staged round of the bitmap out in position order: thread t takes
// words W*t .. W*t+W-1, one block scan of their bit counts gives each thread
// its first output slot, and it writes its positions (the first k of the
// row) to sm.u.c.sel.  Returns the running count.
template <int W>
__device__ __forceinline__ int emit_round(Smem& sm, int64_t w0, int out, int k) {
  uint32_t wd[W];
  const uint32_t* src = sm.u.c.bm + W * threadIdx.x;
  if constexpr (W == 8) {
    const uint4 lo = reinterpret_cast<const uint4*>(src)[0], hi = reinterpret_cast<const uint4*>(src)[1];
    wd[0] = lo.x, wd[1] = lo.y, wd[2] = lo.z, wd[3] = lo.w;
    wd[4] = hi.x, wd[5] = hi.y, wd[6] = hi.z, wd[7] = hi.w;
  } else if constexpr (W == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    wd[0] = v.x, wd[1] = v.y, wd[2] = v.z, wd[3] = v.w;
  } else if constexpr (W == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    wd[0] = v.x, wd[1] = v.y;
  } else {
    wd[0] = *src;
  }
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < W; ++e) cnt += __popc(wd[e]);
  int total;
  int slot = out + block_prefix(cnt, sm, &total);
  const int64_t wb = w0 + W * threadIdx.x;
#pragma unroll
  for (int e = 0; e < W; ++e) {
    uint32_t word = wd[e];
    while (word) {
      const int bit = __ffs(word) - 1;
      word &= word - 1;
      if (slot < k) sm.u.c.sel[slot] = static_cast<int32_t>((wb + e) * 32 + bit);
      ++slot;
    }
  }
  return out + total;
}

// The finish of one row, run by the last of its CTAs.
__device__ __forceinline__ void finish_row(const TopkArgs& a, int64_t row, int64_t V, int64_t ventries, const Crossing& c,
                           Smem& sm) {
  const uint32_t* bits = a.bits + row * a.bits_ld;
  uint32_t* ties = a.ties + row * a.bits_ld;
  const int lane = threadIdx.x & 31;
  const int64_t nwords = (V + 31) >> 5;
  const uint32_t dstar = static_cast<uint32_t>(c.bin);
  int need = a.k - c.above;
  if (threadIdx.x == 0) sm.nx = 0;
  // Words [w0, w0 + kRoundWords) of the bitmap into sm.u.c.bm, eight
  // consecutive words per thread (bits_ld is a multiple of 8: the vectors
  // stay inside the row); words past the row read as zero.
  auto load_round = [&](int64_t w0) {
    const int64_t wb = w0 + kEmitWords * threadIdx.x;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
    if (wb < nwords) {
      lo = __ldcg(reinterpret_cast<const uint4*>(bits + wb));
      hi = __ldcg(reinterpret_cast<const uint4*>(bits + wb + 4));
      const uint32_t left = static_cast<uint32_t>(nwords - wb);
      if (left < 8) {  // the row's last words: the rest of the group is not the row's
        uint32_t v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        for (uint32_t e = left; e < 8; ++e) v[e] = 0u;
        lo = make_uint4(v[0], v[1], v[2], v[3]);
        hi = make_uint4(v[4], v[5], v[6], v[7]);
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(sm.u.c.bm + kEmitWords * threadIdx.x);
    dst[0] = lo;
    dst[1] = hi;
  };
  load_round(0);  // in flight with the candidate loads below
  if (c.in_bin != need) {
    const unsigned ncu = __ldcg(a.cand_count + row);
    int n_eq = 0;
    if (ncu <= static_cast<unsigned>(a.cand_cap)) {
      const int nc = static_cast<int>(ncu);
      const uint32_t* gkey = a.cand_key + row * a.cand_cap;
      const int32_t* gpos = a.cand_idx + row * a.cand_cap;
      const bool staged = nc <= kTopkCandCap;  // a longer list is read from global memory in each pass
      if (staged) {
        for (int i = threadIdx.x; i < nc; i += kThreads) {  // both loads in flight at once
          const int32_t p = __ldcg(gpos + i);
          const uint32_t key = __ldcg(gkey + i);
          const bool ok = p >= 0 && p < V;  // positions come from this row's filter; checked all the same
          sm.u.c.ckey[i] = ok ? key : 0u;
          sm.u.c.cpos[i] = ok ? p : 0;
        }
      }
      // the next 11 bits of the candidates' keys
      for (int i = threadIdx.x; i < 2048; i += kThreads) sm.h.hist[i] = 0;
      if (threadIdx.x == 0) sm.nsmall = 0;
      __syncthreads();
      for_candidates(staged, nc, sm, gkey, gpos, V,
                     [&](uint32_t k, int32_t) { atomicAdd(&sm.h.hist[(k >> 10) & 2047], 1); });
      __syncthreads();
      const Crossing cc = find_crossing(2048, need, sm);
      const uint32_t p22 = (dstar << 11) | static_cast<uint32_t>(cc.bin);  // the crossing bin's top 22 bits
      const int need2 = need - cc.above;
      if (cc.in_bin <= 32) {
        // keys above the bin are taken; the bin's keys are ranked by one warp
        for_candidates(staged, nc, sm, gkey, gpos, V, [&](uint32_t k, int32_t p) {
          const uint32_t k22 = k >> 10;
          if (k22 > p22) mark(sm, p);
          if (k22 == p22) {
            const int slot = atomicAdd(&sm.nsmall, 1);
            if (slot < 32) {
              sm.small_key[slot] = k;
              sm.small_pos[slot] = p;
            }
          }
        });
        __syncthreads();
        if (threadIdx.x < 32) {
          const int nb = min(sm.nsmall, 32);
          const bool has = lane < nb;
          const uint32_t kl = has ? sm.small_key[lane] : 0u;
          const int32_t pl = has ? sm.small_pos[lane] : 0;
          int rank = 0;  // keys of the bin before this one: larger, or equal at a smaller position
          for (int j = 0; j < nb; ++j) {
            const uint32_t kj = __shfl_sync(0xffffffffu, kl, j);
            const int32_t pj = __shfl_sync(0xffffffffu, pl, j);
            rank += (kj > kl) || (kj == kl && pj < pl);
          }
          if (has && rank < need2) mark(sm, pl);
        }
      } else {
        // a crowded bin: one more digit (10 bits) gives the threshold key
        uint32_t thr;
        {
          for (int i = threadIdx.x; i < 1024; i += kThreads) sm.h.hist[i] = 0;
          __syncthreads();
          for_candidates(staged, nc, sm, gkey, gpos, V, [&](uint32_t k, int32_t) {
            if ((k >> 10) == p22) atomicAdd(&sm.h.hist[k & 1023], 1);
          });
          __syncthreads();
          const Crossing c2 = find_crossing(1024, need2, sm);
          thr = (p22 << 10) | static_cast<uint32_t>(c2.bin);
          need = need2 - c2.above;
          n_eq = c2.in_bin;
        }
        const bool all_eq = n_eq == need;  // every key equal to thr is taken
        for_candidates(staged, nc, sm, gkey, gpos, V, [&](uint32_t k, int32_t p) {
          if (k > thr || (k == thr && all_eq)) mark(sm, p);
          if (k == thr && !all_eq) atomicOr(ties + (p >> 5), 1u << (p & 31));
        });
        if (!all_eq) take_ties(ties, nwords, need, sm);
      }
    } else {
      // the candidate list overflowed: the same digits counted over the row's scores
      const uint32_t thr =
          resolve_threshold(dstar, V, [&](int64_t i) { return score_key(row_score(a, row, i)); }, sm, &need, &n_eq);
      const bool all_eq = n_eq == need;
      for (int64_t i0 = 0; i0 < V; i0 += kBatch * kThreads) {
        float xv[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int64_t i = i0 + u * kThreads + threadIdx.x;
          xv[u] = i < V ? row_score(a, row, i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int64_t i = i0 + u * kThreads + threadIdx.x;
          const uint32_t k = i < V ? score_key(xv[u]) : 0u;
          const bool in = i < V && (k >> kKeyBinShift) == dstar;
          if (in && (k > thr || (k == thr && all_eq))) mark(sm, static_cast<int32_t>(i));
          const unsigned em = __ballot_sync(0xffffffffu, in && k == thr && !all_eq);
          if (lane == 0 && em) atomicOr(ties + ((i - lane) >> 5), em);
        }
      }
      if (!all_eq) take_ties(ties, nwords, need, sm);
    }
  }
  __syncthreads();
  const int nx = min(sm.nx, kMaxTopk);  // selected positions past the first round
  // Read the bitmap out in position order, rounds of kRoundWords words from
  // shared memory: eight consecutive words per thread, one block scan per
  // round.  Later rounds (rows longer than 65536 entries) are loaded here and
  // get their selected candidates from the list.
  int out = 0;
  const int k = a.k;
  for (int64_t w0 = 0; w0 < nwords && out < k; w0 += kRoundWords) {
    if (w0 > 0) {
      __syncthreads();  // the previous round is read out
      load_round(w0);
      __syncthreads();
      for (int j = threadIdx.x; j < nx; j += kThreads) {
        const int32_t p = sm.h.xpos[j];
        const int64_t w = (p >> 5) - w0;
        if (w >= 0 && w < kRoundWords) atomicOr(&sm.u.c.bm[w], 1u << (p & 31));
      }
      __syncthreads();
    }
    // a row that fits one round spreads its words over all the threads
    // (fewer set bits to walk per thread); longer rows take 8 words each
    const int64_t left = nwords - w0;
    if (left <= kThreads)
      out = emit_round<1>(sm, w0, out, k);
    else if (left <= 2 * kThreads)
      out = emit_round<2>(sm, w0, out, k);
    else if (left <= 4 * kThreads)
      out = emit_round<4>(sm, w0, out, k);
    else
      out = emit_round<kEmitWords>(sm, w0, out, k);
  }
  __syncthreads();
  int32_t* idx = a.idx_out + row * a.k;
  float* sc = a.score_out ? a.score_out + row * a.k : nullptr;
  for (int j = threadIdx.x; j < a.k; j += kThreads) {
    const int32_t p = j < out ? sm.u.c.sel[j] : -1;
    idx[j] = out_entry(a, row, ventries, p);
    if (sc) sc[j] = p >= 0 ? row_score(a, row, p) + 0.0f : -INFINITY;
  }
}

// The compressor entry of sequence b, 2 channels per thread (m <= 4: the
// m = 8 routine would not fit this kernel's register budget).
__device__ void compress_ride_along(const CompressArgs& c, int b, Smem& sm) {
  const auto sync = [] { __syncthreads(); };
  switch (c.m) {
    case 1: compress_entry<1, 2>(c, b, 0, threadIdx.x, sm.red, sync); break;
    case 2: compress_entry<2, 2>(c, b, 0, threadIdx.x, sm.red, sync); break;
    case 4: compress_entry<4, 2>(c, b, 0, threadIdx.x, sm.red, sync); break;
    default: break;
  }
}

// Grid: x the 4096-key chunks of a row (plus the ride-along column), y the
// queries, z the sequences of problem a0 and then those of problem a1 (a
// second, independent selection over other scores, e.g. the pool's blocks).
__global__ void __launch_bounds__(kThreads, 4)
    topk_kernel(const __grid_constant__ TopkArgs a0, const __grid_constant__ TopkArgs a1, const CompressArgs comp) {
  __shared__ Smem sm;
  pdl_launch_dependents();
  pdl_wait();
  if (comp.B > 0 && blockIdx.x == gridDim.x - 1) {  // the extra column: compressor entries
    if (blockIdx.y == 0) compress_ride_along(comp, blockIdx.z, sm);
    return;
  }
  const bool second = static_cast<int>(blockIdx.z) >= a0.B;
  // a local copy: the compiler keeps the fields it needs in registers (a
  // reference into the parameter space may alias shared memory, and every
  // shared store would force the fields to be read again)
  const TopkArgs a = second ? a1 : a0;
  const int b = static_cast<int>(blockIdx.z) - (second ? a0.B : 0), q = blockIdx.y;
  if (q >= a.Q) return;
  const int64_t row = static_cast<int64_t>(b) * a.Q + q;
  int64_t ventries;
  const int64_t V = row_extent(a, b, q, &ventries);
  if (V <= a.k) {  // every visible entry is selected; the row's first CTA writes it
    if (blockIdx.x != 0) return;
    for (int j = threadIdx.x; j < a.k; j += kThreads) {
      a.idx_out[row * a.k + j] = j < V ? out_entry(a, row, ventries, j) : -1;
      if (a.score_out) a.score_out[row * a.k + j] = j < V ? row_score(a, row, j) + 0.0f : -INFINITY;
    }
    return;
  }
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kItems;
  if (i0 >= V) return;
  const int n_in = static_cast<int>(min(V - i0, static_cast<int64_t>(kItems)));
  // the row's digit counts and the chunk's scores, one bulk copy each on
  // barriers of their own: the crossing search starts once the counts land
  if (threadIdx.x == 0) {
    const int esz = a.bf16_scores ? 2 : 4;
    const uint32_t vbytes = static_cast<uint32_t>((n_in * esz + 15) & ~15);  // score rows are padded to 16 B
    mbar_init(&sm.hist_bar, 1);
    mbar_init(&sm.vals_bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&sm.hist_bar, kKeyBins * 4);
    bulk_load(sm.h.hist, a.hist + row * kKeyBins, kKeyBins * 4, &sm.hist_bar);
    mbar_arrive_expect_tx(&sm.vals_bar, vbytes);
    bulk_load(sm.u.f.vals, reinterpret_cast<const uint8_t*>(a.scores) + (row * a.score_ld + i0) * esz, vbytes,
              &sm.vals_bar);
    sm.n_local = 0;
  }
  __syncthreads();
  if (!__syncthreads_and(mbar_wait(&sm.hist_bar, 0, a.status))) {
    mbar_wait(&sm.vals_bar, 0, a.status);  // no copy of ours stays in flight
    return;
  }
  const Crossing c = find_crossing(kKeyBins, a.k, sm);
  if (!__syncthreads_and(mbar_wait(&sm.vals_bar, 0, a.status))) return;
  const uint32_t dstar = static_cast<uint32_t>(c.bin);
  const bool whole = c.in_bin == a.k - c.above;
  const uint32_t dsel = whole ? dstar : dstar + 1;  // keys with digit >= dsel are selected outright

  // 16 consecutive keys per thread, read as four float4 in a rotated order so
  // that the eight threads of a shared-memory phase hit distinct banks
  const int t = threadIdx.x, lane = t & 31;
  uint32_t smask = 0, cmask = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int jj = (j + (t >> 1)) & 3;
    float xs[4];
    if (a.bf16_scores) {  // the chunk holds bf16 bits: keys 16t .. 16t+15 are 32 bytes
      const uint2 h = reinterpret_cast<const uint2*>(sm.u.f.vals)[4 * t + jj];
      xs[0] = __uint_as_float(h.x << 16), xs[1] = __uint_as_float(h.x & 0xFFFF0000u);
      xs[2] = __uint_as_float(h.y << 16), xs[3] = __uint_as_float(h.y & 0xFFFF0000u);
    } else {
      const float4 x = reinterpret_cast<const float4*>(sm.u.f.vals)[4 * t + jj];
      xs[0] = x.x, xs[1] = x.y, xs[2] = x.z, xs[3] = x.w;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int bit = 4 * jj + e;
      const bool in = 16 * t + bit < n_in;
      const uint32_t d = score_key(xs[e]) >> kKeyBinShift;
      smask |= static_cast<uint32_t>(in && d >= dsel) << bit;
      cmask |= static_cast<uint32_t>(in && !whole && d == dstar) << bit;
    }
  }
  // thread pairs (2u, 2u+1) make bitmap word u of the chunk
  const uint32_t upper = __shfl_down_sync(0xffffffffu, smask, 1);
  if ((t & 1) == 0 && 16 * t < n_in) {
    const int64_t w = (i0 >> 5) + (t >> 1);
    a.bits[row * a.bits_ld + w] = smask | (upper << 16);
    a.ties[row * a.bits_ld + w] = 0u;
  }
  if (__any_sync(0xffffffffu, cmask != 0)) {
    const int cnt = __popc(cmask);
    const int incl = warp_incl_scan(cnt);
    int base = 0;
    if (lane == 31) base = atomicAdd(&sm.n_local, incl);
    int slot = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
    while (cmask) {
      const int bit = __ffs(cmask) - 1;
      cmask &= cmask - 1;
      if (slot < kLocalCap) {
        const float v = a.bf16_scores
                            ? __uint_as_float(static_cast<uint32_t>(
                                                  reinterpret_cast<const unsigned short*>(sm.u.f.vals)[16 * t + bit])
                                              << 16)
                            : sm.u.f.vals[16 * t + bit];
        sm.u.f.lkey[slot] = score_key(v);
        sm.u.f.lpos[slot] = static_cast<int32_t>(i0 + 16 * t + bit);
      }
      ++slot;
    }
  }
  __syncthreads();
  const int n_local = sm.n_local;
  const unsigned cap = static_cast<unsigned>(a.cand_cap);
  if (n_local > kLocalCap) {
    // this CTA's candidates overflowed its local list: the row's count is
    // raised past the cap, so the finish counts from the scores.  A maximum,
    // not an add, so that many overflowing CTAs of one row cannot wrap the
    // count below the cap (the adds below sum to at most the row's length).
    if (threadIdx.x == 0) atomicMax(a.cand_count + row, cap + 1u);
  } else if (n_local > 0) {
    if (threadIdx.x == 0) sm.cand_base = atomicAdd(a.cand_count + row, static_cast<unsigned>(n_local));
    __syncthreads();
    // unsigned throughout: slots at or past the cap are dropped, whatever the count holds
    const unsigned base = sm.cand_base;
    for (int j = threadIdx.x; j < n_local; j += kThreads) {
      if (base < cap && static_cast<unsigned>(j) < cap - base) {
        a.cand_key[row * a.cand_cap + base + j] = sm.u.f.lkey[j];
        a.cand_idx[row * a.cand_cap + base + j] = sm.u.f.lpos[j];
      }
    }
  }
  // The last CTA of the row to get here finishes it: the barrier orders this
  // CTA's writes before thread 0's release, and its acquire (with the
  // barrier after it) orders the other CTAs' writes before the finish reads.
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned n_ctas = static_cast<unsigned>((V + kItems - 1) / kItems);
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(a.row_done + row) : "memory");
    sm.last = prev == n_ctas - 1;
  }
  __syncthreads();
  if (!sm.last) return;
  finish_row(a, row, V, ventries, c, sm);
}

}  // namespace

bool topk_can_carry_compress(int m) { return m == 1 || m == 2 || m == 4; }

int64_t topk_bits_ld(int64_t n_cap) { return ((n_cap + 31) / 32 + kEmitWords - 1) / kEmitWords * kEmitWords; }

// The larger of a sixteenth of the row and four times k (the crossing digit,
// a quarter octave of scores, holds a small fraction of a long row, or a few
// times k where k is a large part of it), at most the row, in whole 256-entry
// steps within the staged size and the largest list.  Past the list a row is
// resolved from its scores.
int topk_cand_cap(int64_t n_cap, int k) {
  int64_t c = n_cap / 16 > 4 * static_cast<int64_t>(k) ? n_cap / 16 : 4 * static_cast<int64_t>(k);
  c = c < n_cap ? c : n_cap;
  c = (c + 255) / 256 * 256;
  return static_cast<int>(c < kTopkCandCap ? kTopkCandCap : (c > kTopkCandCapMax ? kTopkCandCapMax : c));
}

namespace {

// The longest row of a selection: the cache's entries, their blocks, or the
// pool's slots.
int64_t topk_extent(const TopkArgs& a) {
  return a.vis_shift ? (a.n_cap + (int64_t(1) << a.vis_shift) - 1) >> a.vis_shift
                     : (a.pool ? static_cast<int64_t>(a.pool_blocks) * kPoolBlock : a.n_cap);
}

bool topk_args_ok(const TopkArgs& a) {
  return a.cand_cap >= kTopkCandCap && a.cand_cap <= kTopkCandCapMax && !(a.pool && (a.pool_blocks <= 0 || a.vis_shift));
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, const CompressArgs* ride_along, cudaStream_t stream,
                        const TopkArgs* second) {
  if (a.B <= 0 || a.Q <= 0) return cudaSuccess;
  if (!topk_args_ok(a)) return cudaErrorInvalidValue;
  CompressArgs c = {};
  if (ride_along) {
    if (ride_along->mode != 1 || ride_along->B != a.B || !topk_can_carry_compress(ride_along->m) || second)
      return cudaErrorInvalidValue;
    c = *ride_along;
    fill_inv_freq(&c);
  }
  TopkArgs b = {};  // no second problem: B = 0
  int64_t chunks = (topk_extent(a) + kItems - 1) / kItems;
  int q = a.Q;
  if (second && second->B > 0 && second->Q > 0) {
    if (!topk_args_ok(*second)) return cudaErrorInvalidValue;
    b = *second;
    const int64_t c2 = (topk_extent(b) + kItems - 1) / kItems;
    chunks = c2 > chunks ? c2 : chunks;
    q = b.Q > q ? b.Q : q;
  }
  chunks += ride_along ? 1 : 0;
  return launch_pdl(topk_kernel, dim3(static_cast<unsigned>(chunks), q, a.B + b.B), dim3(kThreads), 0, stream, a,
                    b, c);
}

// Clears `bytes` (a multiple of 4, 16-byte aligned) at p: the indexer's and
// the top-k's per-call counters.  A kernel on the programmatic-launch chain
// (it signals its dependents on entry and waits for its predecessor before
// writing), so that the launches around it still overlap, which a memset node
// would not allow.  With a DecodeAppend, B more CTAs (one per sequence) write
// the step's new window row and indexer key into the caches.
namespace {
__global__ void __launch_bounds__(256) zero_kernel(uint32_t* p, const int64_t words, const int zero_blocks,
                                                   const DecodeAppend ap) {
  pdl_launch_dependents();
  pdl_wait();
  if (static_cast<int>(blockIdx.x) >= zero_blocks) {  // one CTA per sequence: its new rows
    const int b = static_cast<int>(blockIdx.x) - zero_blocks;
    const int64_t t = ap.q_pos[b];
    if (t < 0) return;
    const int c = threadIdx.x;
    constexpr int kRowChunks = kDim * 2 / 16, kKeyChunks = kIdxDim / 16;
    if (c < kRowChunks) {
      const uint4* src = reinterpret_cast<const uint4*>(ap.swa_new + static_cast<int64_t>(b) * kDim);
      uint4* dst = reinterpret_cast<uint4*>(ap.swa_ring + (static_cast<int64_t>(b) * ap.W + t % ap.W) * kDim);
      dst[c] = src[c];
    } else if (ap.kI_new && c < kRowChunks + kKeyChunks && (t + 1) % ap.m == 0) {
      const int64_t i = (t + 1) / ap.m - 1;
      if (i < ap.n_cap) {
        const uint4* src = reinterpret_cast<const uint4*>(ap.kI_new + static_cast<int64_t>(b) * kIdxDim);
        uint4* dst = reinterpret_cast<uint4*>(ap.kI + (static_cast<int64_t>(b) * ap.n_cap + i) * kIdxDim);
        dst[c - kRowChunks] = src[c - kRowChunks];
      }
    }
    return;
  }
  const int64_t n4 = words / 4;
  const int64_t step = static_cast<int64_t>(zero_blocks) * blockDim.x;
  uint4* p4 = reinterpret_cast<uint4*>(p);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += step)
    p4[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = n4 * 4 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < words; i += step)
    p[i] = 0u;
}
}  // namespace

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t stream, const DecodeAppend* append) {
  const int64_t words = static_cast<int64_t>(bytes / 4);
  const int rows = append ? append->B : 0;
  if (words <= 0 && rows == 0) return cudaSuccess;
  int64_t blocks = words > 0 ? (words / 4 + 255) / 256 : 0;
  blocks = words <= 0 ? 0 : (blocks < 1 ? 1 : (blocks > 1024 ? 1024 : blocks));
  static_assert(kDim * 2 / 16 + kIdxDim / 16 <= 256, "one CTA copies a sequence's new rows");
  return launch_pdl(zero_kernel, dim3(static_cast<unsigned>(blocks + rows)), dim3(256), 0, stream,
                    static_cast<uint32_t*>(p), words, static_cast<int>(blocks),
                    append ? *append : DecodeAppend{});
}

}  // namespace csa
