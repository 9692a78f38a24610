// Exact top-k of the lightning-indexer scores.  Page "CSA / HCA" (zdszero,
// hca_csa), "CSA：轻压缩 + 稀疏选择" (Top-k over I_{t,:}, all visible entries
// compete, window included); indices reported in ascending entry order
// ("DeepSeek 注意力结构对比" CSA2 section: sorted by position); equal scores
// are broken toward the smaller entry index.
//
// Scores are compared as order-preserving 32-bit keys (keys.cuh).  While it
// scores, the indexer counts each row's keys by their top 11 bits (the
// "digit"), so the digit d* that holds the k-th largest key is known without
// another pass over the row.  One thread-block cluster of G <= 8 CTAs selects
// a row; CTA g owns a contiguous range of the row's 4096-key chunks, whose
// scores it stages on chip with bulk copies (two in flight):
//   filter   a key whose digit is above d* is selected outright: each thread
//            reads 16 consecutive keys and builds half of a 32-bit word of
//            the CTA's position bitmap (on chip for up to 8 chunks).  A key
//            whose digit is d* is a candidate; the CTA lists its candidates
//            in position order.
//   resolve  the candidates' next 11 bits, then (unless the crossing bin is
//            taken whole) their last 10 bits, are counted into the shared
//            memory of the cluster's rank-0 CTA (remote atomic adds) and read
//            back by every CTA after a cluster barrier: every CTA finds the
//            same exact threshold key T and how many keys equal to T are
//            taken (the first ones by position).
//   emit     each CTA counts its keys above T and equal to T and sends both
//            counts to every CTA of the cluster; one more barrier gives each
//            its offset in the row's output and its share of the ties.  It
//            ORs its selected candidates into its bitmap and writes its own
//            positions, ascending, at that offset.
// No CTA waits for another outside the cluster's hardware barriers, and no
// count or list goes through global memory.  A CTA whose candidates outnumber
// its list reads its keys again instead (slower, exact).  When d* alone holds
// exactly the keys still needed, the filter selects all of d* and only the
// counts are exchanged.
//
// A decode step's compressor entry (compress.cuh) can ride along: extra CTAs
// of the same launch compute one sequence's entry each, so their latency
// hides behind the selection.
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
constexpr int kItems = 4096;                // keys per chunk: 16 consecutive keys per thread
constexpr int kChunkWords = kItems / 32;    // bitmap words per chunk
constexpr int kMaxCluster = 16;             // CTAs that share a row (8 where larger clusters are refused)
constexpr int kMaxSlots = 4;                // chunks of scores in flight per CTA
constexpr int kSmemWords = 1024;            // bitmap words a CTA keeps on chip (8 chunks)
constexpr int kListCap = 2 * kThreads;      // candidates a CTA lists (two per thread when ranked)
constexpr int kEmitWords = 4;               // bitmap words a thread reads per emission round
static_assert(kItems == 16 * kThreads, "a thread covers half a bitmap word");
static_assert(kSmemWords == kEmitWords * kThreads, "one emission round covers the on-chip bitmap");
static_assert(kKeyBins == 2048, "first digit: 11 bits");

struct Crossing {
  int bin, above, in_bin;  // the bin, the count in higher bins, the count in it
};

// The dynamic shared memory: this struct, then (at kValsOff) the CTA's score
// slots of kItems fp32 each (bf16 rows fill the first half of a slot): one
// for launches whose CTAs hold one chunk, up to kMaxSlots in flight for
// longer rows.
struct __align__(16) Smem {
  int hist[kKeyBins];             // the row's first-digit counts, then the second-digit counts
  int h3[1024];                   // third-digit counts
  uint32_t bm[kSmemWords];        // this CTA's part of the row's position bitmap
  uint32_t lkey[kListCap];        // its candidates, in position order
  int32_t lpos[kListCap];
  uint4 peer[kMaxCluster];        // per CTA of the cluster: keys above the threshold, keys equal to it
  uint4 res[2];                   // rank 0's results: the second digit's crossing, then the third's
  uint4 lead;                     // rank 0's d*, the count still needed at it, whether it is taken whole
  int wscan[2][kWarps];           // warp totals of block scans (two buffers, used in turn)
  int wsum[kWarps];
  int wval[kWarps];
  float red[kWarps];
  Crossing out;
  uint64_t hist_bar, vals_bar[kMaxSlots];
  uint64_t sum_bar;               // rank 0: one arrival per warp of the cluster per digit (two phases)
  uint64_t res_bar[2];            // rank 0's results landed
  uint64_t peer_bar;              // every CTA's counts landed
};

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
// One barrier: the warps' totals go to buffer `buf`, which the block flips
// after each scan, so that no scan overwrites totals a thread may still be
// reading from the scan before (a barrier of the scan between separates
// them).
__device__ int block_prefix(int cnt, Smem& sm, int* total, int& buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan(cnt);
  if (lane == 31) sm.wscan[buf][warp] = incl;
  __syncthreads();
  int before = 0, sum = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int v = sm.wscan[buf][w];
    before += w < warp ? v : 0;
    sum += v;
  }
  buf ^= 1;
  *total = sum;
  return before + incl - cnt;
}

// Waits (cluster-scope acquire) for a phase of a barrier that other CTAs of
// the cluster complete; gives up after the wait limit (kErrTimeout recorded).
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, unsigned* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns(), limit = wait_limit_ns(status);
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit) {
      record_error(status, kErrTimeout);
      return false;
    }
  }
}

// Block-wide sums of two per-thread counts; every thread gets both.
__device__ void block_sum2(uint32_t* x, uint32_t* y, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t a = *x, b = *y;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    b += __shfl_xor_sync(0xffffffffu, b, off);
  }
  if (lane == 0) {
    sm.wsum[warp] = static_cast<int>(a);
    sm.wval[warp] = static_cast<int>(b);
  }
  __syncthreads();
  a = b = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    a += static_cast<uint32_t>(sm.wsum[w]);
    b += static_cast<uint32_t>(sm.wval[w]);
  }
  __syncthreads();
  *x = a;
  *y = b;
}

// Scanning the counts of nb (1024 or 2048) bins from the top bin down, finds
// the bin in which the running count first reaches `need`.  Thread t holds
// bins nb-1-per*t down to nb-per*(t+1); two barriers.  If the counts never
// reach `need` the result is {0, 0, 0}.
__device__ Crossing find_crossing(const int* bins, int nb, int need, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = nb / kThreads;  // 4 or 8
  const int lo = nb - per * (static_cast<int>(threadIdx.x) + 1);
  int c[8];
  const int4 v0 = *reinterpret_cast<const int4*>(bins + lo + per - 4);
  const int4 v1 = per == 8 ? *reinterpret_cast<const int4*>(bins + lo) : make_int4(0, 0, 0, 0);
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

// One bulk async copy global -> shared completing on `bar` (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Score i of a row (fp32, or bf16 bits widened exactly).
__device__ __forceinline__ float row_score(const TopkArgs& a, int64_t row, int64_t i) {
  if (a.bf16_scores)
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(a.scores) +
                                                      row * a.score_ld + i))
                           << 16);
  return __ldg(a.scores + row * a.score_ld + i);
}

// Score i of a staged chunk.
__device__ __forceinline__ float staged_score(const float* vals, bool bf16, int i) {
  return bf16 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const unsigned short*>(vals)[i]) << 16)
              : vals[i];
}

// Calls f(key, bit) for the 16 keys 16t .. 16t+15 of a staged chunk (bit =
// key - 16t), read as four 16-byte vectors (fp32) in a rotated order so that
// the eight threads of a shared-memory phase hit distinct banks.
template <class F>
__device__ __forceinline__ void visit16(const float* vals, bool bf16, F f) {
  const int t = threadIdx.x;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int jj = (j + (t >> 1)) & 3;
    float xs[4];
    if (bf16) {  // keys 16t .. 16t+15 are 32 bytes
      const uint2 h = reinterpret_cast<const uint2*>(vals)[4 * t + jj];
      xs[0] = __uint_as_float(h.x << 16), xs[1] = __uint_as_float(h.x & 0xFFFF0000u);
      xs[2] = __uint_as_float(h.y << 16), xs[3] = __uint_as_float(h.y & 0xFFFF0000u);
    } else {
      const float4 x = reinterpret_cast<const float4*>(vals)[4 * t + jj];
      xs[0] = x.x, xs[1] = x.y, xs[2] = x.z, xs[3] = x.w;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) f(score_key(xs[e]), 4 * jj + e);
  }
}

// The number of keys of the row: its visible entries; or their blocks
// (vis_shift); or, with a pool, its valid slots: the pool holds
// nb = min(pool_blocks, ceil(V/8)) ascending blocks, all entries visible but
// those of block ceil(V/8)-1 past V, which can only be the pool's last.
// *ventries receives V.
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

// Grid: x the G CTAs of a row's cluster, y the queries, z the sequences of
// problem a0 and then those of problem a1 (a second, independent selection
// over other scores, e.g. the pool's blocks), then the ride-along CTAs (one
// compressor entry each).  Every CTA of a cluster shares y and z, so a row
// that needs no selection is left by the whole cluster at once, and every
// decision between two cluster barriers is taken on values that all its CTAs
// hold alike.
constexpr size_t kValsOff = (sizeof(Smem) + 127) / 128 * 128;

// kMulti: some rows of the launch give a CTA more than one chunk; without
// it every CTA holds at most one (and the kernel carries none of the code of
// the longer rows, a smaller instruction footprint for the common launches).
template <bool kMulti>
__global__ void __launch_bounds__(kThreads, 4)
    topk_kernel(const __grid_constant__ TopkArgs a0, const __grid_constant__ TopkArgs a1, const CompressArgs comp,
                const int G, const int slot_shift) {
  extern __shared__ __align__(128) uint8_t topk_smem[];
  Smem& sm = *reinterpret_cast<Smem*>(topk_smem);
  float* const vbase = reinterpret_cast<float*>(topk_smem + kValsOff);
  pdl_launch_dependents();
  pdl_wait();
  const int zsel = a0.B + a1.B;
  if (static_cast<int>(blockIdx.z) >= zsel) {  // ride-along: one compressor entry per CTA
    const int64_t s =
        (static_cast<int64_t>(blockIdx.z - zsel) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    if (s < comp.B) compress_ride_along(comp, static_cast<int>(s), sm);
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
  const int t = threadIdx.x;
  const int g = blockIdx.x;  // the rank in the cluster
  const bool bf16 = a.bf16_scores != 0;
  const int esz = bf16 ? 2 : 4;
  const uint8_t* srow = reinterpret_cast<const uint8_t*>(a.scores) + row * a.score_ld * esz;
  // The barriers, and the loads that do not depend on the row's extent (a
  // q_pos read): the row's first-digit counts and, when every CTA holds one
  // chunk (chunk g), that chunk's scores as far as the score row reaches.
  uint32_t spec_bytes = 0;  // thread 0: bytes of chunk g loaded ahead
  if (t == 0) {
    mbar_init(&sm.hist_bar, 1);
    for (int i = 0; i < kMaxSlots; ++i) mbar_init(&sm.vals_bar[i], 1);
    mbar_init(&sm.sum_bar, G * kWarps);
    mbar_init(&sm.res_bar[0], 1);
    mbar_init(&sm.res_bar[1], 1);
    mbar_init(&sm.peer_bar, 1);
    fence_mbar_init();
    // the bytes other CTAs will store here (a result not sent leaves its phase open)
    mbar_arrive_expect_tx(&sm.res_bar[0], 16);
    mbar_arrive_expect_tx(&sm.res_bar[1], 16);
    mbar_arrive_expect_tx(&sm.peer_bar, 16 * G);
    mbar_arrive_expect_tx(&sm.hist_bar, kKeyBins * 4);
    bulk_load(sm.hist, a.hist + row * kKeyBins, kKeyBins * 4, &sm.hist_bar);
    if (!kMulti) {
      const int64_t len = min(static_cast<int64_t>(kItems), a.score_ld - static_cast<int64_t>(g) * kItems);
      if (len > 0) {  // score rows are padded to 16 bytes
        spec_bytes = static_cast<uint32_t>((len * esz + 15) & ~int64_t(15));
        mbar_arrive_expect_tx(&sm.vals_bar[0], spec_bytes);
        bulk_load(vbase, srow + static_cast<int64_t>(g) * kItems * esz, spec_bytes, &sm.vals_bar[0]);
      }
    }
  }
  // this CTA's own copies have landed (before it leaves early)
  const auto own_copies_landed = [&] {
    if (t == 0) {
      mbar_wait(&sm.hist_bar, 0, a.status);
      if (spec_bytes) mbar_wait(&sm.vals_bar[0], 0, a.status);
    }
  };
  int64_t ventries;
  const int64_t V = row_extent(a, b, q, &ventries);
  if (V <= a.k) {  // every visible entry is selected; the cluster's first CTA writes the row
    own_copies_landed();
    if (g != 0) return;
    for (int j = t; j < a.k; j += kThreads) {
      a.idx_out[row * a.k + j] = j < V ? out_entry(a, row, ventries, j) : -1;
      if (a.score_out) a.score_out[row * a.k + j] = j < V ? row_score(a, row, j) + 0.0f : -INFINITY;
    }
    return;
  }
  // this CTA's chunks [c0, c0 + nmine) and keys [i_lo, i_hi)
  const int64_t nch = (V + kItems - 1) / kItems;
  const int64_t cpc = (nch + G - 1) / G;
  const int64_t c0 = min(static_cast<int64_t>(g) * cpc, nch);
  const int nmine = static_cast<int>(min(c0 + cpc, nch) - c0);
  const int64_t i_lo = c0 * kItems;
  const int64_t i_hi = nmine > 0 ? min(i_lo + static_cast<int64_t>(nmine) * kItems, V) : i_lo;
  const bool resident = !kMulti || cpc == 1;  // the CTA's only chunk stays staged in slot 0 throughout
  // the CTA's bitmap words: on chip, or (ranges of more than 8 chunks) the row's global scratch
  uint32_t* bm = cpc * kChunkWords <= kSmemWords ? sm.bm : a.bits + row * a.bits_ld + c0 * kChunkWords;
  auto chunk_len = [&](int j) { return static_cast<int>(min(V - (c0 + j) * kItems, static_cast<int64_t>(kItems))); };
  const int nslot = 1 << slot_shift;
  auto vals = [&](int slot) { return vbase + slot * kItems; };
  auto issue = [&](int slot, int j) {  // score rows are padded to 16 bytes
    const uint32_t bytes = static_cast<uint32_t>((chunk_len(j) * esz + 15) & ~15);
    mbar_arrive_expect_tx(&sm.vals_bar[slot], bytes);
    bulk_load(vals(slot), srow + (c0 + j) * kItems * esz, bytes, &sm.vals_bar[slot]);
  };
  if (kMulti && t == 0)
    for (int j = 0; j < nslot && j < nmine; ++j) issue(j, j);  // (one chunk a CTA: loading since the start)
  for (int i = t; i < 1024; i += kThreads) sm.h3[i] = 0;
  // rank 0's results, before they come: read alike by every CTA should a wait give up
  if (t < 2) sm.res[t] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  // A wait that gives up (status recorded) leaves garbage behind but changes
  // no barrier: every CTA still takes every cluster barrier the cluster takes.
  bool ok = __syncthreads_and(mbar_wait(&sm.hist_bar, 0, a.status));
  const Crossing c = find_crossing(sm.hist, kKeyBins, a.k, sm);
  const uint32_t dstar = static_cast<uint32_t>(c.bin);
  const int need = a.k - c.above;
  const bool whole = c.in_bin == need;
  for (int i = t; i < kKeyBins; i += kThreads) sm.hist[i] = 0;  // now the second-digit counts
  if (g == 0 && t == 0) sm.lead = make_uint4(dstar, static_cast<uint32_t>(need), whole, 0u);
  if (G > 1) cluster_arrive();  // barriers set up, counts cleared, rank 0's first digit published

  // ---- filter: outright selections and candidates.  A CTA with one chunk
  // keeps both as masks of each thread's 16 keys in registers; with more,
  // the selections go to the bitmap and the candidates to the list.
  const uint32_t dsel = whole ? dstar : dstar + 1;  // keys with digit >= dsel are selected outright
  uint32_t n_out = 0;                               // this thread's outright selections
  uint32_t r_sel = 0, r_cand = 0;                   // one chunk: this thread's selections and candidates
  int n_cand = 0;                                   // the CTA's candidates
  int sb = 0;                                       // the block scans' buffer
  for (int j = 0; j < nmine; ++j) {
    const int slot = j & (nslot - 1);
    const int n_in = chunk_len(j);
    ok = __syncthreads_and(mbar_wait(&sm.vals_bar[slot], static_cast<uint32_t>(j >> slot_shift) & 1u, a.status)) && ok;
    uint32_t smask = 0, cmask = 0;
    visit16(vals(slot), bf16, [&](uint32_t key, int bit) {
      const bool in = 16 * t + bit < n_in;
      const uint32_t d = key >> kKeyBinShift;
      smask |= static_cast<uint32_t>(in && d >= dsel) << bit;
      cmask |= static_cast<uint32_t>(in && !whole && d == dstar) << bit;
    });
    n_out += __popc(smask);
    if (resident) {
      r_sel = smask, r_cand = cmask;
      break;  // the chunk stays staged
    }
    // thread pairs (2u, 2u+1) make word u of the chunk
    const uint32_t upper = __shfl_down_sync(0xffffffffu, smask, 1);
    if ((t & 1) == 0 && 16 * t < n_in) bm[j * kChunkWords + (t >> 1)] = smask | (upper << 16);
    if (!whole) {
      int total;
      int s = n_cand + block_prefix(__popc(cmask), sm, &total, sb);  // position order
      while (cmask) {
        const int bit = __ffs(cmask) - 1;
        cmask &= cmask - 1;
        if (s < kListCap) {
          sm.lkey[s] = score_key(staged_score(vals(slot), bf16, 16 * t + bit));
          sm.lpos[s] = static_cast<int32_t>(i_lo + static_cast<int64_t>(j) * kItems + 16 * t + bit);
        }
        ++s;
      }
      n_cand += total;
    }
    __syncthreads();  // the slot is read
    if (t == 0 && j + nslot < nmine) issue(slot, j + nslot);
  }
  // Whether the resolution runs is rank 0's decision (equal to this CTA's
  // own unless a copy gave up waiting); the crossings are rank 0's.
  uint32_t ldstar = dstar;
  int lneed = need;
  bool lwhole = whole;
  if (G > 1) {
    cluster_wait();  // every CTA of the cluster is set up
    const uint4 l = dsmem_ld_u32x4(dsmem_addr(&sm.lead, 0));
    ldstar = l.x, lneed = static_cast<int>(l.y), lwhole = l.z != 0;
  }
  const bool listed = n_cand <= kListCap;
  // f(key, position) for each of this CTA's candidates: from the masks
  // (one chunk), the list, or (a list that overflowed) the scores again
  auto for_cands = [&](auto f) {
    if (resident) {
      uint32_t m = r_cand;
      while (m) {
        const int bit = __ffs(m) - 1;
        m &= m - 1;
        f(score_key(staged_score(vals(0), bf16, 16 * t + bit)), static_cast<int32_t>(i_lo + 16 * t + bit));
      }
      return;
    }
    if (listed) {
      for (int i = t; i < n_cand; i += kThreads) f(sm.lkey[i], sm.lpos[i]);
      return;
    }
    for (int64_t i = i_lo + t; i < i_hi; i += kThreads) {
      const uint32_t key = score_key(row_score(a, row, i));
      if ((key >> kKeyBinShift) == ldstar) f(key, static_cast<int32_t>(i));
    }
  };
  // One digit of the candidates' keys counted into rank 0's bins, which
  // alone finds the crossing bin and sends it to every CTA.  G > 1: each add
  // is a remote asynchronous add that completes 4 bytes of rank 0's sum_bar,
  // and each warp arrives there announcing its adds (no fence on the way); a
  // CTA whose list overflowed adds plainly and arrives after a barrier with
  // release order instead (its adds could outgrow a transaction count).
  auto resolve = [&](int* bins, int nb, int phase, int need_at, auto bin_of, auto result) -> uint4 {
    if (G == 1) {
      for_cands([&](uint32_t key, int32_t) {
        const int bin = bin_of(key);
        if (bin >= 0) atomicAdd(bins + bin, 1);
      });
      __syncthreads();
      return result(find_crossing(bins, nb, need_at, sm));
    }
    const uint32_t b0 = dsmem_addr(bins, 0), sbar = dsmem_addr(&sm.sum_bar, 0);
    if (resident || listed) {
      uint32_t mine = 0;
      for_cands([&](uint32_t key, int32_t) {
        const int bin = bin_of(key);
        if (bin < 0) return;
        red_async_add_u32(b0 + 4u * static_cast<uint32_t>(bin), 1u, sbar);
        ++mine;
      });
      const uint32_t wn = __reduce_add_sync(0xffffffffu, mine);
      if ((t & 31) == 0) mbar_arrive_expect_tx_remote(sbar, 4u * wn);
    } else {
      for_cands([&](uint32_t key, int32_t) {
        const int bin = bin_of(key);
        if (bin >= 0) dsmem_red_add_u32(b0 + 4u * static_cast<uint32_t>(bin), 1u);
      });
      __syncthreads();
      if ((t & 31) == 0) mbar_arrive_remote(sbar);  // orders the block's adds before it
    }
    if (g == 0) {
      ok = __syncthreads_and(mbar_wait_cl(&sm.sum_bar, static_cast<uint32_t>(phase), a.status)) && ok;
      const uint4 r = result(find_crossing(bins, nb, need_at, sm));
      // (test fault: the first result is never sent; every CTA's wait gives up)
      if (t < G && !(phase == 0 && test_fault(a.status, kFaultTopk)))
        st_async_v4(dsmem_addr(&sm.res[phase], t), r, dsmem_addr(&sm.res_bar[phase], t));
    }
    ok = __syncthreads_and(mbar_wait_cl(&sm.res_bar[phase], 0, a.status)) && ok;
    return sm.res[phase];
  };

  // ---- resolve: the exact threshold key among the candidates
  uint32_t thr = ldstar << kKeyBinShift;  // selected: keys >= thr (all_eq), else keys > thr and the first ties
  int need_eq = 0;
  bool all_eq = true;
  if (!lwhole) {
    // the next 11 bits: res.x the crossing bin's top 22 bits, .y the count still needed, .z whole bin
    const uint4 r2 = resolve(
        sm.hist, 2048, 0, lneed, [&](uint32_t key) { return static_cast<int>((key >> 10) & 2047u); },
        [&](const Crossing& cc) {
          const int need2 = lneed - cc.above;
          return make_uint4((ldstar << 11) | static_cast<uint32_t>(cc.bin), static_cast<uint32_t>(need2),
                            cc.in_bin == need2, 0u);
        });
    const uint32_t p22 = r2.x;
    thr = p22 << 10;
    if (r2.z == 0) {  // the last 10 bits: res.x the threshold key, .y the ties taken, .z all of them
      const uint4 r3 = resolve(
          sm.h3, 1024, 1, static_cast<int>(r2.y), [&](uint32_t key) { return (key >> 10) == p22 ? static_cast<int>(key & 1023u) : -1; },
          [&](const Crossing& c3) {
            const int q3 = static_cast<int>(r2.y) - c3.above;
            return make_uint4((p22 << 10) | static_cast<uint32_t>(c3.bin), static_cast<uint32_t>(q3),
                              c3.in_bin == q3, 0u);
          });
      thr = r3.x;
      need_eq = static_cast<int>(r3.y);
      all_eq = r3.z != 0;
    }
  }

  // ---- counts: keys above the threshold and keys equal to it, sent to every CTA.
  // One chunk: each thread's selected keys and ties as masks, whose counts one
  // block scan gives both for the exchange and for the output slots.
  uint32_t strict = r_sel, eqm = 0, above = n_out, eq = 0;
  int pre_s = 0, pre_e = 0;
  if (resident) {
    if (!lwhole) {
      uint32_t m = r_cand;
      while (m) {
        const int bit = __ffs(m) - 1;
        m &= m - 1;
        const uint32_t key = score_key(staged_score(vals(0), bf16, 16 * t + bit));
        if (all_eq ? key >= thr : key > thr)
          strict |= 1u << bit;
        else if (!all_eq && key == thr)
          eqm |= 1u << bit;
      }
    }
    int total;  // (a chunk's counts stay below 2^16)
    const int packed = block_prefix(__popc(strict) | (__popc(eqm) << 16), sm, &total, sb);
    pre_s = packed & 0xFFFF, pre_e = packed >> 16;
    above = static_cast<uint32_t>(total & 0xFFFF), eq = static_cast<uint32_t>(total) >> 16;
  } else {
    if (!lwhole)
      for_cands([&](uint32_t key, int32_t) {
        above += all_eq ? key >= thr : key > thr;
        eq += !all_eq && key == thr;
      });
    block_sum2(&above, &eq, sm);
  }
  if (G > 1) {
    if (t < G) st_async_v4(dsmem_addr(&sm.peer[g], t), make_uint4(above, eq, 0u, 0u), dsmem_addr(&sm.peer_bar, t));
    // the CTAs stay until every one has sent its last message (below, before leaving)
    cluster_arrive_relaxed();
    ok = __syncthreads_and(mbar_wait_cl(&sm.peer_bar, 0, a.status)) && ok;
  } else {
    if (t == 0) sm.peer[0] = make_uint4(above, eq, 0u, 0u);
    __syncthreads();
  }
  // this CTA's first output slot, and how many of its keys equal to thr it
  // takes (a row's counts stay below 2^31)
  int off = 0, quota = 0, eq_before = 0;
#pragma unroll
  for (int r = 0; r < kMaxCluster; ++r) {
    if (r < G) {
      const int A = static_cast<int>(sm.peer[r].x), E = static_cast<int>(sm.peer[r].y);
      const int take = all_eq ? 0 : min(max(need_eq - eq_before, 0), E);
      off += r < g ? A + take : 0;
      quota = r == g ? take : quota;
      eq_before += E;
    }
  }
  int32_t* idx = a.idx_out + row * a.k;
  float* sc = a.score_out ? a.score_out + row * a.k : nullptr;
  if (resident) {  // ---- emit: this thread's selected keys and its first ties, in order
    int take = min(max(quota - pre_e, 0), __popc(eqm));
    uint32_t sel = strict;
    for (; take > 0; --take) {
      const uint32_t low = eqm & (0u - eqm);
      sel |= low;
      eqm ^= low;
    }
    int s = off + pre_s + min(pre_e, quota);
    while (sel) {
      const int bit = __ffs(sel) - 1;
      sel &= sel - 1;
      if (s >= 0 && s < a.k) {
        idx[s] = out_entry(a, row, ventries, static_cast<int32_t>(i_lo + 16 * t + bit));
        if (sc) sc[s] = staged_score(vals(0), bf16, 16 * t + bit) + 0.0f;
      }
      ++s;
    }
    if (!ok || nmine == 0) own_copies_landed();  // no copy of ours stays in flight past the CTA
    if (G > 1) cluster_wait();
    return;
  }

  // ---- emit (several chunks): selected candidates into the bitmap, then the bitmap in order
  auto mark = [&](int64_t pos) { atomicOr(bm + ((pos - i_lo) >> 5), 1u << (pos & 31)); };
  if (!lwhole) {
    if (listed) {  // list order is position order: ranks among the keys equal to thr
      const int i0 = 2 * t;
      const bool v0 = i0 < n_cand, v1 = i0 + 1 < n_cand;
      const uint32_t k0 = v0 ? sm.lkey[i0] : 0u, k1 = v1 ? sm.lkey[i0 + 1] : 0u;
      const bool e0 = v0 && !all_eq && k0 == thr, e1 = v1 && !all_eq && k1 == thr;
      int total;
      const int r0 = block_prefix(static_cast<int>(e0) + static_cast<int>(e1), sm, &total, sb);
      if (v0 && (all_eq ? k0 >= thr : (k0 > thr || (e0 && r0 < quota)))) mark(sm.lpos[i0]);
      if (v1 && (all_eq ? k1 >= thr : (k1 > thr || (e1 && r0 + static_cast<int>(e0) < quota))))
        mark(sm.lpos[i0 + 1]);
    } else {  // the keys again, chunk by chunk: 16 consecutive keys per thread
      int ranked = 0;
      for (int j = 0; j < nmine; ++j) {
        const int n_in = chunk_len(j);
        const int64_t base = i_lo + static_cast<int64_t>(j) * kItems + 16 * t;
        uint32_t sel = 0, eqm = 0;
        auto take = [&](uint32_t key, int bit) {
          const bool in = 16 * t + bit < n_in && (key >> kKeyBinShift) == ldstar;
          sel |= static_cast<uint32_t>(in && (all_eq ? key >= thr : key > thr)) << bit;
          eqm |= static_cast<uint32_t>(in && !all_eq && key == thr) << bit;
        };
#pragma unroll 4
        for (int e = 0; e < 16; ++e) take(16 * t + e < n_in ? score_key(row_score(a, row, base + e)) : 0u, e);
        int total;
        int r = ranked + block_prefix(__popc(eqm), sm, &total, sb);
        while (eqm) {
          const int bit = __ffs(eqm) - 1;
          eqm &= eqm - 1;
          if (r < quota) sel |= 1u << bit;
          ++r;
        }
        ranked += total;
        while (sel) {
          const int bit = __ffs(sel) - 1;
          sel &= sel - 1;
          mark(base + bit);
        }
      }
    }
  }
  __syncthreads();
  // the bitmap in position order: four consecutive words per thread, one
  // block scan per round of 1024 words
  const int64_t nw = (i_hi - i_lo + 31) >> 5;
  int64_t run = off;
  for (int64_t w0 = 0; w0 < nw; w0 += kEmitWords * kThreads) {
    const int64_t wb = w0 + kEmitWords * t;
    uint32_t wd[kEmitWords];
    if (wb + kEmitWords <= nw) {
      const uint4 v = *reinterpret_cast<const uint4*>(bm + wb);
      wd[0] = v.x, wd[1] = v.y, wd[2] = v.z, wd[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < kEmitWords; ++e) wd[e] = wb + e < nw ? bm[wb + e] : 0u;
    }
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < kEmitWords; ++e) cnt += __popc(wd[e]);
    int total;
    int64_t s = run + block_prefix(cnt, sm, &total, sb);
#pragma unroll
    for (int e = 0; e < kEmitWords; ++e) {
      uint32_t word = wd[e];
      while (word) {
        const int bit = __ffs(word) - 1;
        word &= word - 1;
        const int64_t pos = i_lo + (wb + e) * 32 + bit;
        if (s >= 0 && s < a.k) {
          idx[s] = out_entry(a, row, ventries, static_cast<int32_t>(pos));
          if (sc) sc[s] = row_score(a, row, pos) + 0.0f;
        }
        ++s;
      }
    }
    run += total;
  }
  if (!ok && t == 0) {  // no copy of ours stays in flight past the CTA
    mbar_wait(&sm.hist_bar, 0, a.status);
    for (int j = max(0, nmine - nslot); j < nmine; ++j)
      mbar_wait(&sm.vals_bar[j & (nslot - 1)], static_cast<uint32_t>(j >> slot_shift) & 1u, a.status);
  }
  if (G > 1) cluster_wait();
}

}  // namespace

bool topk_can_carry_compress(int m) { return m == 1 || m == 2 || m == 4; }

int64_t topk_bits_ld(int64_t n_cap) { return ((n_cap + 31) / 32 + 7) / 8 * 8; }

namespace {

// The longest row of a selection: the cache's entries, their blocks, or the
// pool's slots.
int64_t topk_extent(const TopkArgs& a) {
  return a.vis_shift ? (a.n_cap + (int64_t(1) << a.vis_shift) - 1) >> a.vis_shift
                     : (a.pool ? static_cast<int64_t>(a.pool_blocks) * kPoolBlock : a.n_cap);
}

bool topk_args_ok(const TopkArgs& a) { return !(a.pool && (a.pool_blocks <= 0 || a.vis_shift)); }

// The largest cluster the device schedules with the kernel's largest shared
// memory (16, else 8); sets the kernel's attributes on first use per device.
// 0 if the attributes are refused.
int max_cluster() {
  constexpr int kDevices = 64;
  static int cached[kDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kDevices && cached[dev] > 0) return cached[dev];
  const size_t smem_max = kValsOff + size_t(kMaxSlots) * kItems * 4;
  for (auto k : {topk_kernel<false>, topk_kernel<true>})
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_max)) !=
        cudaSuccess)
      return 0;
  int g = 8;
  if (cudaFuncSetAttribute(topk_kernel<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
      cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kMaxCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kMaxCluster, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_max;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, topk_kernel<true>, &cfg) == cudaSuccess && n > 0) g = kMaxCluster;
  }
  cudaGetLastError();  // a refused size is not an error of a launch
  if (dev >= 0 && dev < kDevices) cached[dev] = g;
  return g;
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
    fill_rope(&c);
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
  // one CTA per chunk up to the largest cluster; longer rows give each CTA
  // several, streamed through up to kMaxSlots slots
  const int gmax = max_cluster();
  if (gmax <= 0) return cudaErrorInvalidValue;
  const int G = static_cast<int>(chunks < 1 ? 1 : (chunks > gmax ? gmax : chunks));
  const int64_t cpc = (chunks + G - 1) / G;
  const int slot_shift = cpc <= 1 ? 0 : (cpc == 2 ? 1 : 2);
  const int64_t per_z = static_cast<int64_t>(G) * q;
  const int64_t extra = ride_along ? (c.B + per_z - 1) / per_z : 0;
  const int64_t z = static_cast<int64_t>(a.B) + b.B + extra;
  if (z > 65535) return cudaErrorInvalidValue;
  const size_t smem = kValsOff + (size_t(1) << slot_shift) * kItems * 4;
  return launch_pdl_cluster(slot_shift == 0 ? topk_kernel<false> : topk_kernel<true>,
                            dim3(static_cast<unsigned>(G), q, static_cast<unsigned>(z)), dim3(kThreads), smem, stream,
                            static_cast<unsigned>(G), a, b, c, G, slot_shift);
}

// Clears `bytes` (a multiple of 4, 16-byte aligned) at p: the indexer's and
// the top-k's per-call counters.  A kernel on the programmatic-launch chain
// (it signals its dependents on entry and waits for its predecessor before
// writing), so that the launches around it still overlap, which a memset node
// would not allow.  With a DecodeAppend, B more CTAs (one per sequence, the
// grid's first, so that they are dispatched before the zeroing CTAs) write
// the step's new window row and indexer key into the caches; the key
// compressor (`key`, ring mode, B > 0) runs on warps 4..7 of those CTAs.
namespace {
__global__ void __launch_bounds__(256, 2) zero_kernel(uint32_t* p, const int64_t words, const int zero_blocks,
                                                   const DecodeAppend ap, const CompressArgs key) {
  // dependents start only after this wait: its predecessor has then
  // completed, so a dependent may read before its own wait whatever this
  // kernel does not write (the indexer's early key tiles)
  pdl_wait();
  pdl_launch_dependents();
  const int seq_blocks = static_cast<int>(gridDim.x) - zero_blocks;
  if (static_cast<int>(blockIdx.x) < seq_blocks) {  // one CTA per sequence: its new rows
    __shared__ float red[4], xch[kIdxDim];
    const int b = static_cast<int>(blockIdx.x);
    const int c = threadIdx.x;
    constexpr int kRowChunks = kDim * 2 / 16, kKeyChunks = kIdxDim / 16, kKeyThread0 = 128;
    static_assert(kRowChunks + kKeyChunks <= kKeyThread0 && kKeyThread0 + kIdxDim == 256, "threads' roles");
    if (c >= kKeyThread0) {  // (reads the position itself, with its other loads)
      if (key.B > 0)
        index_key_entry_wide_m(key, b, c - kKeyThread0, red, xch, [] { named_bar_sync(1, kIdxDim); });
      return;
    }
    const int64_t t = ap.q_pos[b];
    if (t < 0) return;
    if (c < kRowChunks) {
      if (!ap.swa_new) return;
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
  const int64_t zb = static_cast<int64_t>(blockIdx.x) - seq_blocks;
  uint4* p4 = reinterpret_cast<uint4*>(p);
  for (int64_t i = zb * blockDim.x + threadIdx.x; i < n4; i += step) p4[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = n4 * 4 + zb * blockDim.x + threadIdx.x; i < words; i += step) p[i] = 0u;
}
}  // namespace

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t stream, const DecodeAppend* append,
                        const CompressArgs* keys) {
  const int64_t words = static_cast<int64_t>(bytes / 4);
  const int rows = append ? append->B : 0;
  CompressArgs k = {};  // B = 0: no key compressor
  if (keys) {
    if (!append || keys->mode != 1 || keys->B != append->B || keys->m != append->m) return cudaErrorInvalidValue;
    k = *keys;
    fill_rope(&k);
  }
  if (words <= 0 && rows == 0) return cudaSuccess;
  int64_t blocks = words > 0 ? (words / 4 + 255) / 256 : 0;
  blocks = words <= 0 ? 0 : (blocks < 1 ? 1 : (blocks > 1024 ? 1024 : blocks));
  static_assert(kDim * 2 / 16 + kIdxDim / 16 <= 256, "one CTA copies a sequence's new rows");
  return launch_pdl(zero_kernel, dim3(static_cast<unsigned>(blocks + rows)), dim3(256), 0, stream,
                    static_cast<uint32_t*>(p), words, static_cast<int>(blocks),
                    append ? *append : DecodeAppend{}, k);
}

}  // namespace csa
