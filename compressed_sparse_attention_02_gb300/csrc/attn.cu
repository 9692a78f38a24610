// Shared-KV sparse MQA with a joint softmax over [window rows || selected
// compressed rows || sink].  Page "CSA / HCA" (zdszero, hca_csa), section
// "设计：近处看原文，远处看摘要" (o_{t,i} equation; the sink enters the shared
// denominator only); gather semantics "DeepSeek-V4 的 KV 压缩：从删 token 误解到
// 预算检索" §9.5–9.6; flash-style running max / running sum with a fused sink
// ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §19.3).
//
// A query's rows are shared by `split` CTAs (1, 2 or 4; a thread-block
// cluster when above 1) or `gsplit` CTAs (split-KV, merged by a second
// kernel), each holding all 64 heads and a contiguous slice of the query's
// row set.  The 64 heads share every K=V row, so both products run with the
// gathered rows on the MMA's M side (M = 128: an N = 64 product costs the
// same ~52 clocks at M = 64 as at M = 128, so smaller tiles would double the
// first product's cost):
//   S^T[row, head]  = KV_tile[128 x 512] . Q^T[512 x 64]   (K-major A and B)
//   O^T[ch, head]  += V^T[512 x 128] . P^T[128 x 64]       (MN-major A and B)
// The same 128-byte-swizzled KV tile in shared memory is the K-major A
// operand of the first product and the MN-major A operand of the second.
// S^T (64 TMEM columns) and O^T (4 x 64 columns, one per 128-channel block)
// live in TMEM.
//
// The CTA is warp-specialised and pipelined within its one KV buffer (the
// 64 KiB Q tile and a 128 KiB tile leave no room for a second):
//   warp 8 (one thread) issues the MMAs: S of a tile granule by granule (a
//     granule is a 128-channel quarter of the tile) as each lands, then,
//     once P is written, O one 128-channel block at a time, committing each
//     block to its own barrier;
//   warps 0-7 gather the next tile's granule g into the buffer as soon as
//     O has finished with channel block g (16-byte cp.async per row piece,
//     or, for a tile of 128 consecutive present rows of the window buffer or
//     of a dense cache run, two TMA boxes), so the gather overlaps the O
//     product and the next S product overlaps the gather; then they run the
//     softmax of the tile: a thread owns one tile row (its TMEM lane) and 32
//     heads.  The reference maximum of a head moves only when a logit
//     exceeds it by more than 2^8, found by a barrier OR over the threads'
//     checks; only then are the per-head tile maxima reduced across rows and
//     O^T rescaled.  Row sums are kept per thread and reduced once after the
//     last tile.  The final division uses the same reference, so the result
//     does not depend on when it moved.
// Every wait is bounded; a wait that gives up raises a CTA-wide abort flag
// that ends every other wait, so all roles leave their loops together.
//
// With split > 1 each CTA ends with its slice's (O^T, reference max, sum) per
// head.  The cluster combines them through distributed shared memory: every
// CTA reads all CTAs' maxima and sums, scales its own O^T by its share of the
// joint softmax (sink included once), stages it as fp32 in its (now free) KV
// buffer, and then sums one channel slice over the cluster's buffers and
// writes it.  With gsplit > 1 the slices' raw O^T and (max, sum) go to the
// workspace and attn_combine_kernel merges them.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kWorkers = 256;             // warps 0-7: gather, softmax, epilogue
constexpr int kMmaWarp = kWorkers / 32;   // warp 8: TMA of Q and MMA issue
constexpr int kThreads = kWorkers + 32;
constexpr uint32_t kBarWorkers = 1;       // named barrier over the workers
constexpr int kTileRows = 128;
constexpr int kGranules = 4;              // 128-channel quarters of a tile
constexpr uint32_t kKVBytes = kTileRows * kDim * 2;       // 128 KiB: [8 blocks][128 rows][128 B]
constexpr uint32_t kPBytes = kTileRows * kHeads * 2;      // 16 KiB: [128 rows][64 heads]
constexpr uint32_t kKVBlock = kTileRows * 128;            // 16 KiB per 64-channel block of KV
constexpr uint32_t kGranuleBytes = 2 * kKVBlock;          // 32 KiB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 64;                            // O^T columns start here
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleSlack = 8.0f;                     // log2 units

constexpr uint32_t kQBytes = kHeads * kDim * 2;           // 64 KiB: [8 blocks][64 heads][128 B]
constexpr uint32_t kQBlock = kHeads * 128;                // 8 KiB per 64-channel block of Q
constexpr int HW = kHeads / 2;                            // heads per worker warp (two share a TMEM quadrant)
constexpr int kMaxSplit = 4;  // the exchange below needs 2*(split-1)/split of 192 KiB
static_assert(kKVBytes == kHeads * kDim * 4, "the KV buffer stages the fp32 partial output");
static_assert(kQBytes + kKVBytes == 192 * 1024, "the output exchange uses the Q and KV buffers");

// How a tile's rows reach shared memory.
enum : int { kTileGather = 0, kTileTmaWindow = 1, kTileTmaEntries = 2 };

constexpr int kNumBars = 5 + 3 * kGranules;
constexpr size_t kLutBytes = 256 * 4;  // FP4 rows: byte -> two bf16 E2M1 values
constexpr size_t kSmemBytes = 1024 + kQBytes + kKVBytes + kPBytes + kMaxTopk * 4 + 4 * kHeads * 4 +
                              4 * kHeads * 4 + 2 * kMaxSplit * kHeads * 4 + kNumBars * 8 + 16 + kLutBytes;

// Inverse partial RoPE of the output: channel chn's pair (D-R+2j, D-R+2j+1)
// is turned by -t * theta^(-2j/R).  rope_angle gives (sin, cos) of t *
// theta^(-2j/R) (the fixed-point angle of rope_sincos: positions reach
// 2^20); inverse_rope turns one value, exchanging it with the pair's other
// lane (adjacent lanes of a warp: every lane of the warp must call it).
__device__ __forceinline__ void rope_angle(int chn, int64_t t, const AttnArgs& a, float* s, float* c) {
  rope_sincos(t, a.rope_turns[(chn - (kDim - kRope)) >> 1], s, c);
}

__device__ __forceinline__ float inverse_rope(float x, int chn, float s, float c) {
  const float partner = __shfl_xor_sync(0xffffffffu, x, 1);
  // pair (u, v) -> (u cos + v sin, -u sin + v cos)
  return (chn & 1) ? fmaf(x, c, -partner * s) : fmaf(x, c, partner * s);
}

// Two E2M1 codes (the low nibble first) as a bf16 pair: the E2M1 grid
// 0, 0.5, 1, 1.5, 2, 3, 4, 6 with the sign in bit 3.
__device__ __forceinline__ uint32_t e2m1_pair_bf16(uint32_t byte) {
  constexpr uint16_t kMag[8] = {0x0000, 0x3F00, 0x3F80, 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0};
  const uint32_t lo = kMag[byte & 7u] | ((byte & 8u) << 12), hi = kMag[(byte >> 4) & 7u] | ((byte & 0x80u) << 8);
  return lo | (hi << 16);
}

// An E4M3 scale as a bf16 pair (E4M3 values are exact in bf16).
__device__ __forceinline__ __nv_bfloat162 e4m3_bf16x2(uint32_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
  const float f = __half2float(__half(h));
  return __floats2bfloat162_rn(f, f);
}

// bf16 bits of x rounded to nearest, ties to even, by integer arithmetic
// (the conversion instruction is slow here; x finite or NaN, which stays NaN).
__device__ __forceinline__ uint32_t bf16_bits_rn(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
  return (u & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC0u : r;
}

// 2^x (MUFU; subnormal results flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled block.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Reduce-scatter of 32 per-thread values across a warp: afterwards lane l
// holds in v[0] the reduction over all 32 lanes of value l.
template <bool kMax>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 16 >> step;
    const int mask = 16 >> step;
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, mask);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

// The row set of one query, [window rows || selected (or, dense, all
// visible) entries], and the addresses of its rows.  Plain values and
// force-inlined functions: nothing of it lives in local memory, which (with
// the shared memory this kernel takes) would be an L2 round trip per access.
struct RowSet {
  const uint16_t* swa;     // this sequence's window buffer: [W] ring or [swa_len] linear rows
  const uint16_t* kv;      // this sequence's bf16 cache
  const uint8_t* kv_fp4;   // this sequence's FP4 cache
  uint32_t sel;            // the compacted selection (shared-memory address)
  int64_t swa_rel0;        // linear window: buffer row of window row 0
  int64_t swa_len;
  int W, swa_mode, n_swa, n_rows, slot0, dense;
};

// Address of window row j (0 <= j < n_swa), null if the window buffer lacks it.
__device__ __forceinline__ const uint16_t* window_row(const RowSet& s, int j) {
  if (s.swa_mode == 0) {
    const int slot = s.slot0 + j < s.W ? s.slot0 + j : s.slot0 + j - s.W;  // j < n_swa <= W
    return s.swa + static_cast<int64_t>(slot) * kDim;
  }
  const int64_t rr = s.swa_rel0 + j;
  return rr >= 0 && rr < s.swa_len ? s.swa + rr * kDim : nullptr;
}

// Address of row j of the row set (null: absent or past the set); an FP4
// entry's address is returned for its bytes.
template <bool kFp4>
__device__ __forceinline__ const uint16_t* row_addr(const RowSet& s, int j) {
  if (j < s.n_swa) return window_row(s, j);
  if (j >= s.n_rows) return nullptr;
  int64_t e = j - s.n_swa;
  if (!s.dense) {
    int32_t v;
    asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(s.sel + 4u * static_cast<uint32_t>(j - s.n_swa)));
    e = v;
  }
  if constexpr (kFp4) return reinterpret_cast<const uint16_t*>(s.kv_fp4 + e * kFp4Entry);
  return s.kv + e * kDim;
}

// Whether the tile of rows r0 .. r0+127 loads by TMA: all present and
// consecutive in one buffer, i.e. the whole window (linear buffer, or the
// W = 128 ring, whose slots then hold exactly the window, in slot order,
// which the softmax does not see), or a run of consecutive entries of a
// dense bf16 cache.  y: the TMA row coordinate.
struct TileLoad {
  int mode;
  int32_t y;
};
template <bool kFp4>
__device__ __forceinline__ TileLoad tile_load(const RowSet& s, int r0, int r_hi, const AttnArgs& a) {
  TileLoad t = {kTileGather, 0};
  if (r0 + kTileRows > r_hi) return t;
  if (r0 + kTileRows <= s.n_swa) {
    if (!a.tma_swa) return t;
    if (s.swa_mode == 0) {
      if (s.W == kTileRows && s.n_swa == kTileRows) t.mode = kTileTmaWindow;
      return t;
    }
    const int64_t rr0 = s.swa_rel0 + r0;
    if (rr0 >= 0 && rr0 + kTileRows <= s.swa_len) {
      t.mode = kTileTmaWindow;
      t.y = static_cast<int32_t>(rr0);
    }
    return t;
  }
  if (!kFp4 && s.dense && a.tma_kv && r0 >= s.n_swa) {
    t.mode = kTileTmaEntries;
    t.y = r0 - s.n_swa;
  }
  return t;
}

// A bounded wait that also ends when another thread of the CTA has raised
// the abort flag; a wait that runs out records kErrTimeout and raises it.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned* status) {
  constexpr uint32_t kSleepNs = 20000;  // the thread wakes when the phase completes
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns(), limit = wait_limit_ns(status);
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit) {
      record_error(status, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// The query's 64 x 512 bf16 rows into eight 128-byte-swizzled 64-channel
// blocks, on q_full (one thread).
__device__ __forceinline__ void load_q(const CUtensorMap& tm_q, uint8_t* q_s, int64_t row_q, uint64_t* q_full) {
  prefetch_tensormap(&tm_q);
  mbar_arrive_expect_tx(q_full, kQBytes);
#pragma unroll
  for (int blk = 0; blk < 8; ++blk)
    tma_load_2d(q_s + blk * kQBlock, &tm_q, blk * 64, static_cast<int32_t>(row_q * kHeads), q_full);
}

// kFp4: the compressed rows are FP4 entries (a.kv_fp4); a template
// argument, so that the bf16 kernel carries none of that code.
template <bool kFp4>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_swa,
                       const __grid_constant__ CUtensorMap tm_kv, const AttnArgs a, const int split,
                       const int gsplit) {
  extern __shared__ uint8_t smem_raw[];
  // (offset from smem_raw, not an integer round trip: the pointers keep the
  // shared address space, so their accesses are shared-memory instructions)
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* q_s = base;                                          // [8 blocks][64 heads][128 B]
  uint8_t* kv_s = q_s + kQBytes;                                // [8 blocks][128 rows][128 B]
  uint8_t* p_s = kv_s + kKVBytes;                               // [128 rows][64 heads] bf16
  int32_t* sel_s = reinterpret_cast<int32_t*>(p_s + kPBytes);
  float* red_s = reinterpret_cast<float*>(sel_s + kMaxTopk);    // [4 row quadrants][64]
  float* m_ref = red_s + 4 * kHeads;                            // running reference max (log2 units)
  float* l_sum = m_ref + kHeads;                                // the denominator after the last tile
  float* alpha = l_sum + kHeads;                                // per-head rescale factor
  float* fin = alpha + kHeads;                                  // the sink logit
  float* ml_s = fin + kHeads;  // [split][2][64]: every slice's reference max and sum (split > 1)
  uint64_t* bars = reinterpret_cast<uint64_t*>(ml_s + 2 * kMaxSplit * kHeads);
  uint64_t* q_full = bars;          // the Q tile (TMA)
  uint64_t* recv_bar = bars + 1;    // incoming output slices (split > 1)
  uint64_t* s_full = bars + 2;      // S of the tile is in TMEM (MMA commit)
  uint64_t* p_full = bars + 3;      // P of the tile is written (every worker)
  uint64_t* drain_bar = bars + 4;   // MMAs in flight when a wait gave up
  uint64_t* landed = bars + 5;      // [4] granule gathered by the workers (every worker)
  uint64_t* tma_bar = landed + kGranules;  // [4] granule loaded by TMA (bytes)
  uint64_t* o_done = tma_bar + kGranules;  // [4] O has read channel block g (MMA commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);            // [0] n_sel, [1] rescale, [2] abort
  uint32_t* lut = reinterpret_cast<uint32_t*>(flags + 3);        // [256] (FP4 rows)
  volatile int* abort_flag = flags + 2;

  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool worker = tid < kWorkers;
  if (split > 1) {
    if (tid == 0) {  // expects the (split-1) output slices the peers will send
      mbar_init(recv_bar, 1);
      mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((split - 1) * (kKVBytes / split)));
      fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive();  // waited on before the first access to a peer
  }
  // Without a.early: wait before any global access and before TMEM is
  // taken.  With it, the barriers are set up and Q (an input no kernel of the
  // chain writes) starts loading first.
  if (!a.early) pdl_wait();
  const int quad = warp & 3;         // TMEM lane quadrant == 32 tile rows
  const int hw0 = (warp >> 2) * HW;  // first head of this worker warp
  // the query's row set is cut into `split` slices combined in the cluster,
  // or `gsplit` slices combined by attn_combine_kernel (one of them is 1)
  const int slices = split > 1 ? split : gsplit;
  const int qi = blockIdx.x / slices;
  const int rank = blockIdx.x % slices;  // == the CTA's rank in its cluster when split > 1
  const int b = blockIdx.y;
  const int64_t row_q = static_cast<int64_t>(b) * a.Q + qi;
  const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[row_q]) : a.pos_base + qi;

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, kWorkers);
    mbar_init(drain_bar, 1);
    for (int g = 0; g < kGranules; ++g) {
      mbar_init(landed + g, kWorkers);
      mbar_init(tma_bar + g, 1);
      mbar_init(o_done + g, 1);
    }
    fence_mbar_init();
    flags[1] = 0;
    flags[2] = 0;
  }
  if (a.early) {  // Q by TMA now; TMEM and the predecessors' outputs after the wait
    __syncthreads();
    if (warp == kMmaWarp && lane == 0) load_q(tm_q, q_s, row_q, q_full);
    pdl_wait();
  }
  // This thread's share of the selection, read right after the dependency
  // wait so that its latency overlaps the set-up (and the q_pos read)
  constexpr int kIdxPer = (kMaxTopk + kThreads - 1) / kThreads;
  const int per = (a.k + kThreads - 1) / kThreads;  // <= kIdxPer
  const int lo = min(a.k, tid * per), hi = min(a.k, lo + per);
  int32_t pv[kIdxPer];
  if (!a.dense) {
    const int32_t* ig = a.idx + row_q * a.k;
#pragma unroll
    for (int u = 0; u < kIdxPer; ++u) pv[u] = lo + u < hi ? ig[lo + u] : -1;
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  if (tid < kHeads) {
    m_ref[tid] = -INFINITY;
    l_sum[tid] = 0.f;
    fin[tid] = a.sink[tid] * kLog2e;  // the sink logit until the epilogue
  }

  const int n_swa = static_cast<int>(t < 0 ? 0 : min(static_cast<int64_t>(a.W), t + 1));
  RowSet rs;
  rs.swa = a.swa + static_cast<int64_t>(b) * (a.swa_mode == 0 ? a.W : a.swa_len) * kDim;
  rs.kv = a.kv + static_cast<int64_t>(b) * a.n_cap * kDim;
  rs.kv_fp4 = a.kv_fp4 + static_cast<int64_t>(b) * a.n_cap * kFp4Entry;
  rs.sel = smem_u32(sel_s);
  {
    const int64_t swa_first = t - n_swa + 1;  // position of window row 0
    const int64_t swa_pos0 = a.swa_mode == 1 ? (a.swa_pos0 ? a.swa_pos0[b] : a.swa_pos0_base) : 0;
    rs.swa_rel0 = swa_first - swa_pos0;
    rs.slot0 = a.swa_mode == 0 ? static_cast<int>(swa_first % a.W) : 0;  // its ring slot
  }
  rs.swa_len = a.swa_len;
  rs.W = a.W;
  rs.swa_mode = a.swa_mode;
  rs.n_swa = n_swa;
  rs.dense = a.dense;

  // Compact the selected entries (drop -1, flag out-of-range indices).
  // Dense (HCA): the rows are the visible entries 0 .. V(t)-1, no list.
  if (!a.dense) {
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kIdxPer; ++u) {
      const int32_t v = pv[u];
      if (lo + u >= hi) break;
      if (v >= 0 && v < a.n_cap) ++cnt;
      else if (v != -1 && rank == 0) record_error(a.status, kErrIndexRange);
    }
    int x = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    __shared__ int wtot[kThreads / 32];
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    int before = x - cnt;
    for (int w = 0; w < warp; ++w) before += wtot[w];
#pragma unroll
    for (int u = 0; u < kIdxPer; ++u) {
      const int32_t v = pv[u];
      if (lo + u >= hi) break;
      if (v >= 0 && v < a.n_cap) sel_s[before++] = v;
    }
    if (tid == kThreads - 1) flags[0] = before;
  }
  __syncthreads();
  int n_sel;
  if (a.dense) {
    int64_t V = t >= 0 ? (t + 1) / a.m : 0;
    if (V > a.n_cap) {
      if (tid == 0 && rank == 0) record_error(a.status, kErrIndexRange);
      V = a.n_cap;
    }
    n_sel = static_cast<int>(V);
  } else {
    n_sel = flags[0];
  }
  const int n_rows = n_swa + n_sel;
  // this CTA's slice of the row set [window rows || selected rows]
  const int per_cta = (n_rows + slices - 1) / slices;
  const int r_lo = min(n_rows, rank * per_cta);
  const int r_hi = min(n_rows, r_lo + per_cta);
  const int n_tiles = (r_hi - r_lo + kTileRows - 1) / kTileRows;
  const float scale2 = a.sm_scale * kLog2e;

  rs.n_rows = n_rows;
  if constexpr (kFp4)
    if (worker) lut[tid] = e2m1_pair_bf16(tid);  // one entry per worker
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tlane = tmem + (static_cast<uint32_t>(quad * 32) << 16);  // this warp's TMEM quadrant

  if (warp == kMmaWarp) {
    // ---------------- Q by TMA, then the MMAs of every tile ----------------
    if (lane == 0) {
      if (!a.early) load_q(tm_q, q_s, row_q, q_full);
      // (waited for even without a tile: the epilogue may reuse the Q buffer)
      bool ok = wait_or_abort(q_full, 0, abort_flag, a.status);
      constexpr uint32_t idesc_s = instr_desc(kTileRows, kHeads, 1, 1, 0, 0);  // bf16, K-major A/B
      constexpr uint32_t idesc_o = instr_desc(kTileRows, kHeads, 1, 1, 1, 1);  // bf16, MN-major A/B
      const uint32_t kvb = smem_u32(kv_s), qb = smem_u32(q_s), pb = smem_u32(p_s);
      int n_gather = 0, n_tma = 0;  // tiles so far of each kind: the phases of landed / tma_bar
      // test fault: the first tile's S is never announced (the workers' waits give up)
      const bool skip_s = test_fault(a.status, kFaultAttn);
      for (int j = 0; j < n_tiles && ok; ++j) {
        const bool tma = tile_load<kFp4>(rs, r_lo + j * kTileRows, r_hi, a).mode != kTileGather;
        const uint32_t par = static_cast<uint32_t>(tma ? n_tma++ : n_gather++) & 1u;
        // S^T = KV . Q^T, granule by granule as each lands (8 MMAs of K = 16 each)
        for (int g = 0; g < kGranules && ok; ++g) {
          ok = wait_or_abort(tma ? tma_bar + g : landed + g, par, abort_flag, a.status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            const int blk = 2 * g + bb;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc(kvb + blk * kKVBlock + kk * 32, 16, 1024, kSwizzle128B);
              const uint64_t bd = smem_desc(qb + blk * kQBlock + kk * 32, 16, 1024, kSwizzle128B);
              mma_f16(tmem, ad, bd, idesc_s, (blk | kk) ? 1u : 0u);
            }
          }
        }
        if (!ok) break;
        if (!(skip_s && j == 0)) tc_commit(s_full);
        ok = wait_or_abort(p_full, static_cast<uint32_t>(j) & 1u, abort_flag, a.status);
        if (!ok) break;
        tc_fence_after();
        // O^T += V^T . P^T, one 128-channel block (8 K-steps of 16 rows) per commit
#pragma unroll
        for (int g = 0; g < kGranules; ++g) {
#pragma unroll
          for (int ks = 0; ks < kTileRows / 16; ++ks) {
            const uint64_t ad = smem_desc(kvb + 2 * g * kKVBlock + ks * 2048, kKVBlock, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(pb + ks * 2048, kPBytes, 1024, kSwizzle128B);
            mma_f16(tmem + kOCol + g * 64, ad, bd, idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(o_done + g);
        }
      }
      if (!ok) {  // whatever was issued finishes before TMEM is released
        tc_commit(drain_bar);
        mbar_wait(drain_bar, 0, a.status);
      }
    }
    __syncwarp();
  } else {
    // ---------------- workers: gather, softmax ----------------
    const int r = quad * 32 + lane;  // TMEM lane == tile row of this thread's softmax
    float lpart[HW];                 // this thread's partial row sums of its warp's heads
#pragma unroll
    for (int h = 0; h < HW; ++h) lpart[h] = 0.f;
    int tma_tiles = 0;           // thread 0: TMA tiles issued (the phase of tma_bar)
    uint32_t tma_pending = 0u;   // thread 0: granules of its last TMA tile
    // Tile j's rows into the KV buffer, granule g once O has read channel
    // block g of the previous tile (wait_o, phase opar).  Gathered tiles:
    // each worker then signals `landed[g]` once its own copies of g are done.
    // A wait of the whole warp taken by its lane 0 alone (the others wait at
    // the shuffle, not on the barrier's shared-memory word, which the tensor
    // cores' operand reads share).
    auto warp_wait = [&](uint64_t* bar, uint32_t par) -> bool {
      bool w = true;
      if (lane == 0) w = wait_or_abort(bar, par, abort_flag, a.status);
      return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    };
    auto gather = [&](int j, bool wait_o, uint32_t opar) -> bool {
      const int r0 = r_lo + j * kTileRows;
      const TileLoad tl = tile_load<kFp4>(rs, r0, r_hi, a);
      const int mode = tl.mode;
      const int32_t y = tl.y;
      if (mode != kTileGather) {
        if (tid == 0) {
          const CUtensorMap* map = mode == kTileTmaWindow ? &tm_swa : &tm_kv;
          const uint32_t par = static_cast<uint32_t>(tma_tiles++) & 1u;
          tma_pending = 0u;
          for (int g = 0; g < kGranules; ++g) {
            if (wait_o && !wait_or_abort(o_done + g, opar, abort_flag, a.status)) return false;
            mbar_arrive_expect_tx(tma_bar + g, kGranuleBytes);
            tma_load_3d(kv_s + 2 * g * kKVBlock, map, 2 * g * 64, y, b, tma_bar + g);
            tma_load_3d(kv_s + (2 * g + 1) * kKVBlock, map, (2 * g + 1) * 64, y, b, tma_bar + g);
            tma_pending = (tma_pending | (1u << g)) | (par << 8);
          }
        }
        return true;
      }
      if constexpr (!kFp4) {
        // thread tid copies 16-byte chunk tid & 7 of block 2g + ((tid >> 3) & 1)
        // of rows (tid >> 4) + 16i: a half-warp covers a row's 256 bytes of
        // the granule.  The warp's 16 rows are looked up once, one per lane
        // (lane l: row 2w + (l & 1) + 16 (l >> 1)), and taken by shuffles: a
        // row's address may need the selection in shared memory, and lookups
        // interleaved with the copies would each wait behind the previous copy.
        const int jl = r0 + 2 * warp + (lane & 1) + 16 * ((lane >> 1) & 7);
        const uint16_t* mine = lane < 16 && jl < r_hi ? row_addr<kFp4>(rs, jl) : nullptr;
        if (lane < 16 && !mine && jl < n_swa && jl < r_hi) record_error(a.status, kErrIndexRange);
        const uint64_t mine_u = reinterpret_cast<uint64_t>(mine);
        const uint16_t* src[kTileRows / 16];
#pragma unroll
        for (int i = 0; i < kTileRows / 16; ++i)
          src[i] = reinterpret_cast<const uint16_t*>(__shfl_sync(0xffffffffu, mine_u, (lane >> 4) + 2 * i));
        const int bb = (tid >> 3) & 1, c = tid & 7;
        for (int g = 0; g < kGranules; ++g) {
          if (wait_o && !warp_wait(o_done + g, opar)) {
            cp_async_wait_pending(0);
            return false;
          }
          const int blk = 2 * g + bb;
          uint8_t* blk_s = kv_s + blk * kKVBlock;
#pragma unroll
          for (int i = 0; i < kTileRows / 16; ++i) {
            uint8_t* dst = blk_s + swz((tid >> 4) + 16 * i, c);
            if (src[i]) cp_async_16_free(dst, src[i] + blk * 64 + c * 8);
            else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
          }
          cp_async_commit();
          if (g > 0) {  // the previous granule's copies of this thread are done
            cp_async_wait_pending(1);
            fence_proxy_async_smem();
            mbar_arrive(landed + g - 1);
          }
        }
      } else {
        // FP4 rows: thread tid takes rows (tid >> 2) + 64i and, in granule g,
        // channels 32*part .. 32*part+31 with part = 4g + (tid & 3) (16 code
        // bytes and 2 scales of the entry; chunks 4*(part&1) .. +3 of block
        // part>>1).  All codes are loaded first, ahead of the O product; the
        // bf16 values (value * scale is exact in bf16) are written once the
        // granule is free.  Window rows (bf16) take the same 64 bytes by cp.async.
        constexpr int kRowsPer = kTileRows * 4 / kWorkers;  // 2
        const uint16_t* src[kRowsPer];
        bool packed[kRowsPer];
        uint4 nib[kGranules][kRowsPer];
        uint32_t scl[kGranules][kRowsPer];
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
          const int jr = r0 + (tid >> 2) + 64 * i;
          src[i] = jr < r_hi ? row_addr<kFp4>(rs, jr) : nullptr;
          if (!src[i] && jr < n_swa && jr < r_hi && (tid & 3) == 0) record_error(a.status, kErrIndexRange);
          packed[i] = src[i] && jr >= n_swa;
          const uint8_t* e = reinterpret_cast<const uint8_t*>(src[i]);
#pragma unroll
          for (int g = 0; g < kGranules; ++g) {
            const int part = 4 * g + (tid & 3);
            nib[g][i] = packed[i] ? __ldg(reinterpret_cast<const uint4*>(e + 16 * part)) : make_uint4(0u, 0u, 0u, 0u);
            scl[g][i] = packed[i] ? __ldg(reinterpret_cast<const unsigned short*>(e + kDim / 2 + 2 * part)) : 0u;
          }
        }
#pragma unroll
        for (int g = 0; g < kGranules; ++g) {
          if (wait_o && !warp_wait(o_done + g, opar)) {
            cp_async_wait_pending(0);
            return false;
          }
          const int part = 4 * g + (tid & 3), pblk = part >> 1, c0 = (part & 1) * 4;
          uint8_t* blk_s = kv_s + pblk * kKVBlock;
#pragma unroll
          for (int i = 0; i < kRowsPer; ++i) {
            const int rr = (tid >> 2) + 64 * i;
            if (src[i] && !packed[i]) {
#pragma unroll
              for (int k = 0; k < 4; ++k) cp_async_16_free(blk_s + swz(rr, c0 + k), src[i] + pblk * 64 + (c0 + k) * 8);
              continue;
            }
            const __nv_bfloat162 s_lo = e4m3_bf16x2(scl[g][i] & 0xFFu), s_hi = e4m3_bf16x2(scl[g][i] >> 8);
            const uint32_t w[4] = {nib[g][i].x, nib[g][i].y, nib[g][i].z, nib[g][i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // chunk k: code bytes 4k .. 4k+3 (8 channels)
              const __nv_bfloat162 sc = k < 2 ? s_lo : s_hi;
              uint32_t o[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint32_t v = lut[(w[k] >> (8 * q)) & 0xFFu];
                const __nv_bfloat162 x = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&v), sc);
                o[q] = *reinterpret_cast<const uint32_t*>(&x);
              }
              *reinterpret_cast<uint4*>(blk_s + swz(rr, c0 + k)) = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
          cp_async_commit();
          if (g > 0) {
            cp_async_wait_pending(1);
            fence_proxy_async_smem();
            mbar_arrive(landed + g - 1);
          }
        }
      }
      cp_async_wait_pending(0);
      fence_proxy_async_smem();
      mbar_arrive(landed + kGranules - 1);
      return true;
    };

    bool ok = n_tiles == 0 || gather(0, false, 0u);
    for (int j = 0; j < n_tiles; ++j) {
      ok = warp_wait(s_full, static_cast<uint32_t>(j) & 1u) && ok;
      if (!named_bar_and(kBarWorkers, kWorkers, ok)) {  // every worker leaves together
        ok = false;
        break;
      }
      __syncwarp();  // converged for the warp-wide TMEM loads
      tc_fence_after();
      // ---- logits of this thread's row (its warp's 32 heads)
      const int jr = r_lo + j * kTileRows + r;
      const bool valid = jr < r_hi && (jr >= n_swa || window_row(rs, jr) != nullptr);
      float l[HW];
      auto load_logits = [&] {
        uint32_t v[32];
        tmem_ld32(tlane + hw0, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < HW; ++h) l[h] = valid ? __uint_as_float(v[h]) * scale2 : -INFINITY;
      };
      load_logits();
      // the warp's heads' reference maxima (m_ref changes only below, between barriers)
      float mref[HW];
#pragma unroll
      for (int h = 0; h < HW; h += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(m_ref + hw0 + h);
        mref[h] = m4.x, mref[h + 1] = m4.y, mref[h + 2] = m4.z, mref[h + 3] = m4.w;
      }
      bool need = false;
#pragma unroll
      for (int h = 0; h < HW; ++h) need |= l[h] > mref[h] + kRescaleSlack;
      if (named_bar_or(kBarWorkers, kWorkers, need)) {
        // ---- a reference maximum moves: per-head tile maxima over the rows
        //      (the reduction consumes l, read again from TMEM afterwards)
        warp_reduce_scatter<true>(l);
        red_s[quad * kHeads + hw0 + lane] = l[0];
        named_bar_sync_any(kBarWorkers, kWorkers);
        if (tid < kHeads) {
          const float tmax = fmaxf(fmaxf(red_s[tid], red_s[kHeads + tid]),
                                   fmaxf(red_s[2 * kHeads + tid], red_s[3 * kHeads + tid]));
          const float mo = m_ref[tid];
          float al = 1.f;
          if (tmax > mo + kRescaleSlack) {  // also taken on the first tile (mo = -inf)
            al = (mo == -INFINITY) ? 0.f : exp2f(mo - tmax);
            m_ref[tid] = tmax;
            if (j > 0 && al != 1.f) flags[1] = 1;
          }
          alpha[tid] = al;
        }
        named_bar_sync_any(kBarWorkers, kWorkers);
        const bool rescale = flags[1] != 0;
#pragma unroll
        for (int h = 0; h < HW; ++h) {
          lpart[h] *= alpha[hw0 + h];
          mref[h] = m_ref[hw0 + h];
        }
        if (rescale) {  // O^T columns of this warp's heads (O of the previous tile is complete)
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
            const uint32_t taddr = tlane + kOCol + blk * 64 + hw0;
            uint32_t v[32];
            tmem_ld32(taddr, v);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) v[h] = __float_as_uint(__uint_as_float(v[h]) * alpha[hw0 + h]);
            tmem_st32(taddr, v);
          }
          tmem_wait_st();
        }
        named_bar_sync_any(kBarWorkers, kWorkers);  // flags[1] and red_s read by every worker
        if (tid == 0) flags[1] = 0;
        __syncwarp();
        load_logits();
      }
      // ---- P = 2^(l - m_ref) as bf16 into the swizzled P tile; partial row sums
      //      (one packed conversion per pair of heads; an invalid row
      //      contributes zeros, whatever its logits and references give)
#pragma unroll
      for (int c = 0; c < HW / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = c * 8 + 2 * i;
          const __nv_bfloat162 pb = __floats2bfloat162_rn(ex2(l[h] - mref[h]), ex2(l[h + 1] - mref[h + 1]));
          const uint32_t u = valid ? *reinterpret_cast<const uint32_t*>(&pb) : 0u;
          lpart[h] += __uint_as_float(u << 16);
          lpart[h + 1] += __uint_as_float(u & 0xFFFF0000u);
          w[i] = u;
        }
        *reinterpret_cast<uint4*>(p_s + swz(r, hw0 / 8 + c)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(p_full);
      // ---- the next tile's rows, granule by granule as O frees them
      if (j + 1 < n_tiles) ok = gather(j + 1, true, static_cast<uint32_t>(j) & 1u);
      __syncwarp();
    }
    // O of the last tile is complete before the epilogue reads TMEM
    if (ok && n_tiles > 0) ok = warp_wait(o_done + kGranules - 1, static_cast<uint32_t>(n_tiles - 1) & 1u);
    cp_async_wait_pending(0);  // no copy of this thread's stays in flight
    if (tid == 0)              // nor a TMA box (bounded, whatever happened to the other waits)
      for (int g = 0; g < kGranules; ++g)
        if (tma_pending & (1u << g)) mbar_wait(tma_bar + g, (tma_pending >> 8) & 1u, a.status);
    __syncwarp();
    // the denominator of each head over the CTA's rows
    warp_reduce_scatter<false>(lpart);
    red_s[quad * kHeads + hw0 + lane] = lpart[0];
    named_bar_sync_any(kBarWorkers, kWorkers);
    if (tid < kHeads)
      l_sum[tid] = (red_s[tid] + red_s[kHeads + tid]) + (red_s[2 * kHeads + tid] + red_s[3 * kHeads + tid]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool live = *abort_flag == 0 && n_tiles > 0;  // TMEM holds this CTA's O^T
  uint16_t* og = a.out + row_q * kHeads * kDim;

  // ---- epilogue: out = sum over the slices s of O_s^T * 2^(m_s - M) / den,
  //      M the joint maximum (sink included), den = sum_s l_s 2^(m_s - M) +
  //      2^(sink*log2e - M).  `factors` gives slice s's factor for head h.
  auto factors = [&](int h, const float* mvals, const float* lvals, int stride, int n, float* out_f) {
    const float sk = fin[h];
    float M = sk;
    for (int s = 0; s < n; ++s) M = fmaxf(M, mvals[s * stride + h]);
    float den = M == -INFINITY ? 0.f : exp2f(sk - M);
    for (int s = 0; s < n; ++s) {
      const float ms = mvals[s * stride + h];
      if (ms != -INFINITY) den += lvals[s * stride + h] * exp2f(ms - M);
    }
    for (int s = 0; s < n; ++s) {
      const float ms = mvals[s * stride + h];
      out_f[s * kHeads + h] = (M == -INFINITY || ms == -INFINITY) ? 0.f : exp2f(ms - M) / den;
    }
    if (a.lse && rank == 0) a.lse[row_q * kHeads + h] = M == -INFINITY ? -INFINITY : (M + log2f(den)) / kLog2e;
  };
  if (gsplit > 1) {
    // this slice's raw O^T and (reference max, sum) per head, fp32, for the
    // combine kernel: for a head, a warp's lanes hold 32 consecutive channels
    float* po = a.part_o + (row_q * gsplit + rank) * kHeads * kDim;
    float* pml = a.part_ml + (row_q * gsplit + rank) * 2 * kHeads;
    if (tid < kHeads) {
      pml[tid] = m_ref[tid];
      pml[kHeads + tid] = l_sum[tid];
    }
    // [64 heads][512] fp32 straight from TMEM to global memory: for a head a
    // warp's lanes hold 32 consecutive channels, so each store is one
    // 128-byte line, and nothing waits for the stores before the CTA exits
    if (worker) {
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        const int chn = blk * 128 + quad * 32 + lane;
        uint32_t v[32];
        if (live) {
          tmem_ld32(tlane + kOCol + blk * 64 + hw0, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] = 0u;
        }
#pragma unroll
        for (int h = 0; h < 32; ++h) po[(hw0 + h) * kDim + chn] = __uint_as_float(v[h]);
      }
    }
  } else if (split == 1) {
    if (tid < kHeads) factors(tid, m_ref, l_sum, 0, 1, alpha);
    __syncthreads();
    // O^T from TMEM straight to the [64 heads][512] bf16 output (for a head, a
    // warp's lanes hold 32 consecutive channels: one 64-byte run per store);
    // nothing waits for the stores before the CTA exits
    if (worker) {
      // this warp's 32 head factors, read before any output store (which
      // the compiler could not otherwise move them past)
      float fa[32];
#pragma unroll
      for (int h = 0; h < 32; h += 4) {
        const float4 f4 = *reinterpret_cast<const float4*>(alpha + hw0 + h);
        fa[h] = f4.x, fa[h + 1] = f4.y, fa[h + 2] = f4.z, fa[h + 3] = f4.w;
      }
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        const int chn = blk * 128 + quad * 32 + lane;
        uint32_t v[32];
        if (live) {
          tmem_ld32(tlane + kOCol + blk * 64 + hw0, v);
          tmem_wait_ld();
        }
        const bool rot = a.inverse_rope && chn - lane >= kDim - kRope;  // warp-uniform
        float rs = 0.f, rc = 1.f;
        if (rot) rope_angle(chn, t, a, &rs, &rc);
#pragma unroll
        for (int h = 0; h < 32; h += 2) {  // one packed conversion per pair of heads
          float o0 = live ? __uint_as_float(v[h]) * fa[h] : 0.f;
          float o1 = live ? __uint_as_float(v[h + 1]) * fa[h + 1] : 0.f;
          if (rot) {
            o0 = inverse_rope(o0, chn, rs, rc);
            o1 = inverse_rope(o1, chn, rs, rc);
          }
          const __nv_bfloat162 ob = __floats2bfloat162_rn(o0, o1);
          const uint32_t u = *reinterpret_cast<const uint32_t*>(&ob);
          og[(hw0 + h) * kDim + chn] = static_cast<uint16_t>(u);
          og[(hw0 + h + 1) * kDim + chn] = static_cast<uint16_t>(u >> 16);
        }
      }
    }
  } else {
    // Channel slice c (cw channels, whole 128-channel blocks) of the output
    // belongs to CTA c.  Each CTA stages its raw O^T for the other CTAs'
    // slices, fp32 [64 heads][cw], in its Q/KV buffers, and one thread sends
    // each to its owner with a bulk copy; every CTA also sends its (max, sum)
    // to all.  The owner scales what it receives and its own share (read from
    // TMEM) by the slices' factors and adds them.  Staging slot of destination
    // o: o or o-1 (skipping this CTA); receiving slot of source s: split-1 +
    // (s or s-1).
    const int cw = kDim / split;
    const uint32_t slab = kKVBytes / split;  // bytes of one slice
    uint8_t* xbuf = q_s;                     // [2*(split-1)][slab], Q and KV buffers in turn
    auto slot = [&](int x) { return x < rank ? x : x - 1; };
    const int own_blk0 = rank * 4 / split, own_blks = 4 / split;
    cluster_wait();  // every CTA of the cluster has started
    if (tid < kHeads) {
      for (int s = 0; s < split; ++s) {
        dsmem_st_f32(dsmem_addr(&ml_s[(rank * 2) * kHeads + tid], s), m_ref[tid]);
        dsmem_st_f32(dsmem_addr(&ml_s[(rank * 2 + 1) * kHeads + tid], s), l_sum[tid]);
      }
    }
    if (worker) {
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        if (blk >= own_blk0 && blk < own_blk0 + own_blks) continue;
        const int chn = blk * 128 + quad * 32 + lane;
        const int owner = chn / cw, c = chn - owner * cw;
        uint32_t v[32];
        if (live) {
          tmem_ld32(tlane + kOCol + blk * 64 + hw0, v);
          tmem_wait_ld();
        }
        float* dst = reinterpret_cast<float*>(xbuf + slot(owner) * slab) + hw0 * cw + c;
#pragma unroll
        for (int h = 0; h < 32; ++h) dst[h * cw] = live ? __uint_as_float(v[h]) : 0.f;
      }
    }
    fence_proxy_async_smem();
    cluster_sync();  // all slices done: (max, sum) delivered, staging complete, receiving slots free
    if (tid == 0) {
      for (int o = 0; o < split; ++o) {
        if (o == rank) continue;
        // in owner o, this CTA's slice lands in receiving slot split-1 + (rank < o ? rank : rank-1)
        const int rslot = (split - 1) + (rank < o ? rank : rank - 1);
        bulk_copy_to_cluster(dsmem_addr(xbuf + rslot * slab, o), xbuf + slot(o) * slab, slab,
                             dsmem_addr(recv_bar, o));
      }
      bulk_commit_group();
    }
    // every slice's factor per head (red_s is free: [split <= 4][64] factors)
    float* fs = red_s;
    if (tid < kHeads) factors(tid, ml_s, ml_s + kHeads, 2 * kHeads, split, fs);
    // own share from TMEM while the slices travel
    float acc[2][32];
    if (worker) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (k >= own_blks) break;
        uint32_t v[32];
        if (live) {
          tmem_ld32(tlane + kOCol + (own_blk0 + k) * 64 + hw0, v);
          tmem_wait_ld();
        }
#pragma unroll
        for (int h = 0; h < 32; ++h) acc[k][h] = live ? __uint_as_float(v[h]) : 0.f;
      }
    }
    const bool got = __syncthreads_and(mbar_wait(recv_bar, 0, a.status));
    if (worker) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (k >= own_blks) break;
        const int chn = (own_blk0 + k) * 128 + quad * 32 + lane;
        const int c = chn - rank * cw;
#pragma unroll
        for (int h = 0; h < 32; ++h) acc[k][h] *= fs[rank * kHeads + hw0 + h];
        for (int s = 0; s < split && got; ++s) {
          if (s == rank) continue;
          const float* src = reinterpret_cast<const float*>(xbuf + (split - 1 + slot(s)) * slab) + hw0 * cw + c;
#pragma unroll
          for (int h = 0; h < 32; ++h) acc[k][h] = fmaf(src[h * cw], fs[s * kHeads + hw0 + h], acc[k][h]);
        }
        const bool rot = a.inverse_rope && chn - lane >= kDim - kRope;  // warp-uniform
        float rs = 0.f, rc = 1.f;
        if (rot) rope_angle(chn, t, a, &rs, &rc);
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float o = rot ? inverse_rope(acc[k][h], chn, rs, rc) : acc[k][h];
          og[(hw0 + h) * kDim + chn] = static_cast<uint16_t>(bf16_bits_rn(o));
        }
      }
    }
    if (tid == 0) bulk_wait_all();  // this CTA's sends have left its shared memory
    cluster_sync();                 // and every CTA has received before any leaves
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The slices of a query split with gsplit > 1 merged: per head, the joint
// maximum M over the slices' reference maxima and the sink (log2 units), the
// denominator 2^(sink - M) + sum_s l_s 2^(m_s - M), and the output
// sum_s O_s 2^(m_s - M) / den (the merge the cluster does on chip).  One CTA
// per query and 8 heads, one warp per head (few CTAs: a launch of one CTA per
// head spent most of its time dispatching them): lane l loads channels
// 16l .. 16l+15 of every slice (up to 4 slices at once, before the factors)
// while its warp reduces the slices' (max, sum), then sums them; the inverse
// RoPE rotates its channel pairs in place.  G is a bound on gsplit (2, 4, 8
// or 16), so that a launch with few slices keeps few registers.
constexpr int kCombineHeads = 8;
template <int G>
__global__ void __launch_bounds__(32 * kCombineHeads) attn_combine_kernel(const AttnArgs a, const int gsplit) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t row_q = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kCombineHeads + warp;  // one warp per head
  const int c0 = 16 * lane;                          // 16 channels per lane
  const float* po = a.part_o + (row_q * gsplit * kHeads + h) * kDim + c0;
  const int64_t slice_ld = static_cast<int64_t>(kHeads) * kDim;
  // up to 4 slices: their outputs do not depend on the factors, so their
  // loads go out first
  constexpr int kPre = G <= 4 ? G : 1;
  float4 o[kPre][4];
  if constexpr (G <= 4) {
#pragma unroll
    for (int s = 0; s < G; ++s)
      if (s < gsplit)
#pragma unroll
        for (int v = 0; v < 4; ++v) o[s][v] = *reinterpret_cast<const float4*>(po + s * slice_ld + 4 * v);
  }
  // the factors: lane s holds slice s's (max, sum); with the sink logit
  // they give each slice's weight exp2(m_s - M) / den
  const float* ml = a.part_ml + row_q * gsplit * 2 * kHeads;
  const float sk = a.sink[h] * kLog2e;
  const float ms = lane < gsplit ? ml[lane * 2 * kHeads + h] : -INFINITY;
  const float ls = lane < gsplit ? ml[lane * 2 * kHeads + kHeads + h] : 0.f;
  float M = fmaxf(sk, ms);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float den = (M == -INFINITY || ms == -INFINITY) ? 0.f : ls * exp2f(ms - M);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  den += M == -INFINITY ? 0.f : exp2f(sk - M);
  const float fl = (M == -INFINITY || ms == -INFINITY) ? 0.f : exp2f(ms - M) / den;
  if (lane == 0 && a.lse) a.lse[row_q * kHeads + h] = M == -INFINITY ? -INFINITY : (M + log2f(den)) / kLog2e;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
  for (int s = 0; s < G; ++s) {
    if (s < gsplit) {
      const float f = __shfl_sync(0xffffffffu, fl, s);
      float4 ov[4];
#pragma unroll
      for (int v = 0; v < 4; ++v)
        ov[v] = G <= 4 ? o[s < kPre ? s : 0][v] : *reinterpret_cast<const float4*>(po + s * slice_ld + 4 * v);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        acc[4 * v + 0] = fmaf(f, ov[v].x, acc[4 * v + 0]);
        acc[4 * v + 1] = fmaf(f, ov[v].y, acc[4 * v + 1]);
        acc[4 * v + 2] = fmaf(f, ov[v].z, acc[4 * v + 2]);
        acc[4 * v + 3] = fmaf(f, ov[v].w, acc[4 * v + 3]);
      }
    }
  }
  if (a.inverse_rope && c0 >= kDim - kRope) {  // pairs (c, c+1): (u, v) -> (u cos + v sin, -u sin + v cos)
    const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[row_q]) : a.pos_base + row_q % a.Q;
#pragma unroll
    for (int pr = 0; pr < 8; ++pr) {
      float rs, rc;
      rope_angle(c0 + 2 * pr, t, a, &rs, &rc);
      const float u = acc[2 * pr], v = acc[2 * pr + 1];
      acc[2 * pr] = fmaf(u, rc, v * rs);
      acc[2 * pr + 1] = fmaf(v, rc, -u * rs);
    }
  }
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162 pr2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&pr2);
  }
  uint4* dst = reinterpret_cast<uint4*>(a.out + (row_q * kHeads + h) * kDim + c0);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// The largest cluster size (a power of two up to kMaxSplit) that the device
// can schedule for this kernel at all, found once per device.
int max_split(int dev) {
  constexpr int kDevices = 64;
  static int cached[kDevices] = {};
  if (dev >= 0 && dev < kDevices && cached[dev] > 0) return cached[dev];
  int split = kMaxSplit;
  for (; split > 1; split /= 2) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split), 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_attn_kernel<false>, &cfg) == cudaSuccess && n > 0) break;
    cudaGetLastError();  // a refused size is not an error of the launch
  }
  if (dev >= 0 && dev < kDevices) cached[dev] = split;
  return split;
}

// CTAs per query: enough that the launch covers about one CTA per SM, at
// most what a cluster allows, a divisor of the 512 channels.
int choose_split(int64_t queries, int sms, int limit) {
  int split = 1;
  while (split < limit && queries * split * 2 <= sms) split *= 2;
  return split;
}

// A 3-D map over bf16 rows of kDim channels, [seqs][rows][kDim], read in
// boxes of one 64-channel block of kTileRows consecutive rows of one
// sequence (128-byte swizzle, the KV tile's layout).
bool encode_rows_map(CUtensorMap* m, PFN_cuTensorMapEncodeTiled_v12000 encode, const uint16_t* base, int64_t rows,
                     int64_t seqs) {
  if (!encode || !base || rows < kTileRows || seqs <= 0) return false;
  cuuint64_t dim[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(seqs)};
  cuuint64_t stride[2] = {static_cast<cuuint64_t>(kDim) * 2, static_cast<cuuint64_t>(rows) * kDim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTileRows), 1};
  cuuint32_t ones[3] = {1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dim, stride, box, ones,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Slices of at most this many tiles take the split-KV form (fp32 partials and
// the merge kernel) rather than a cluster's on-chip merge.
#ifndef CSA_ATTN_GSPLIT_TILES
#define CSA_ATTN_GSPLIT_TILES 3
#endif

cudaError_t launch_sparse_attn(const AttnArgs& args, PFN_cuTensorMapEncodeTiled_v12000 encode, cudaStream_t stream) {
  if (args.B <= 0 || args.Q <= 0) return cudaSuccess;
  AttnArgs a = args;
  // q: [B*Q*64 rows][512 bf16]; a box is one 64-channel block of one query's 64 heads
  CUtensorMap tm_q;
  {
    cuuint64_t dim[2] = {static_cast<cuuint64_t>(kDim),
                         static_cast<cuuint64_t>(a.B) * static_cast<cuuint64_t>(a.Q) * kHeads};
    cuuint64_t stride[1] = {static_cast<cuuint64_t>(kDim) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kHeads)};
    cuuint32_t ones[2] = {1, 1};
    if (!encode || encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.q), dim, stride, box,
                          ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // the window buffer ([B][W] ring or [B][swa_len] linear rows) and, for
  // dense attention over a bf16 cache, the cache: tiles of consecutive rows
  // by TMA (a map that cannot be made leaves those tiles to the gather)
  CUtensorMap tm_swa = {}, tm_kv = {};
  a.tma_swa = encode_rows_map(&tm_swa, encode, a.swa, a.swa_mode == 0 ? a.W : a.swa_len, a.B) ? 1 : 0;
  a.tma_kv = !a.kv_fp4 && a.dense && encode_rows_map(&tm_kv, encode, a.kv, a.n_cap, a.B) ? 1 : 0;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto kernel = a.kv_fp4 ? sparse_attn_kernel<true> : sparse_attn_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int64_t queries = static_cast<int64_t>(a.B) * a.Q;
  const int cluster_max = max_split(dev);
  // With the caller's workspace: split each query's rows over separate CTAs
  // (one wave, at most one slice per 128-row tile of the longest row set, at
  // most what the workspace holds), merged by a second kernel.  Taken when
  // it gives more slices than a cluster holds, or slices of at most 3 tiles;
  // with longer slices the cluster's on-chip merge was measured faster.
  int gsplit = 1;
  if (a.part_o && a.part_ml && a.gsplit_cap >= 2) {
    const int64_t rows_max = a.W + (a.dense ? a.n_cap : a.k);
    int64_t g = sms / queries;
    g = g < a.gsplit_cap ? g : a.gsplit_cap;
    const int64_t tiles = (rows_max + kTileRows - 1) / kTileRows;
    g = g < tiles ? g : tiles;
    if (g >= 2 && (g > cluster_max || (tiles + g - 1) / g <= CSA_ATTN_GSPLIT_TILES)) gsplit = static_cast<int>(g);
  }
  if (gsplit > 1) {
    e = launch_pdl(kernel, dim3(static_cast<unsigned>(a.Q) * gsplit, a.B), dim3(kThreads), kSmemBytes, stream, tm_q,
                   tm_swa, tm_kv, a, 1, gsplit);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(queries), kHeads / kCombineHeads), block(32 * kCombineHeads);
    static_assert(kMaxGSplit == 16, "the merge kernel is instantiated for bounds up to 16");
    if (gsplit <= 2) return launch_pdl(attn_combine_kernel<2>, grid, block, 0, stream, a, gsplit);
    if (gsplit <= 4) return launch_pdl(attn_combine_kernel<4>, grid, block, 0, stream, a, gsplit);
    if (gsplit <= 8) return launch_pdl(attn_combine_kernel<8>, grid, block, 0, stream, a, gsplit);
    return launch_pdl(attn_combine_kernel<16>, grid, block, 0, stream, a, gsplit);
  }
  const int split = choose_split(queries, sms, cluster_max);
  return launch_pdl_cluster(kernel, dim3(static_cast<unsigned>(a.Q) * split, a.B), dim3(kThreads), kSmemBytes,
                            stream, static_cast<unsigned>(split), tm_q, tm_swa, tm_kv, a, split, 1);
}

}  // namespace csa
