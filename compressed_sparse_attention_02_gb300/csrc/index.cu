// Lightning-indexer scores on the 5th-generation tensor cores.
// Page "CSA / HCA" (zdszero, hca_csa), section "CSA：轻压缩 + 稀疏选择",
// equation I_{t,s} = sum_h w_{t,h} ReLU(q^I_{t,h} . K^IComp_s); causal
// visibility "DeepSeek-V4 的 KV 压缩：从删 token 误解到预算检索" §9.8.
//
// The product is computed transposed, S^T = K^I . q^I^T: a tile of 128 keys
// is the MMA's M (one TMEM lane per key), the QPC queries' 64 heads are N, and
// the 128 FP8 channels are K (four kind::f8f6f4 MMAs of K = 32).  Each
// epilogue thread then owns one key and reduces its 64 head scores with the
// head weights and ReLU in registers: no cross-thread reduction.
//
// Persistent grid: exactly the CTAs that fit on the GPU at once, each taking
// an equal contiguous range of the flattened (query group, key tile) space.
// Warp roles (576 threads):
//   warp 0      TMA producer: q^I of each query group it meets (two buffers),
//               and a STAGES-deep ring of 16 KiB K^I tiles (128-byte
//               swizzle, L2 evict-first);
//   warp 1      TMEM owner and MMA issuer (one thread) into NBUF TMEM
//               accumulators, so epilogues of earlier tiles overlap MMAs;
//   warps 2..17 epilogue, four groups of four warps (one query per tile:
//               groups take tiles in turn; four queries: a group per query):
//               tcgen05.ld, weighted ReLU sum (four independent chains),
//               coalesced fp32 score stores for keys visible to the query,
//               and the row's histogram of score-key top digits (used by
//               the top-k to go straight to the digit holding the k-th).
// Every wait is bounded; a timeout records the error, the roles drain their
// own in-flight work and the CTA releases TMEM and exits.
//
// Hierarchical indexer ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §11, and
// §20.1: the candidates are gathered before they are scored).  Full layer:
// the epilogue also takes the maximum over each block of 8 consecutive keys
// (three shuffles: a block is 8 adjacent lanes) and stores it with its own
// first-digit histogram, for the top-k that picks the pool's blocks.
// Reindex layer: a tile is 16 pool blocks instead of 128 consecutive keys;
// the producer loads each block (8 keys, 1 KiB, one 128-byte swizzle atom)
// with its own TMA box into the tile's atom slot, so the MMA and the epilogue
// run unchanged, and scores are stored by pool slot.
#include <cuda_bf16.h>

#include "keys.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kTileKeys = 128;
constexpr uint32_t kSfBytes = 512;  // FP4: a key tile's scale atom, a query's scale record
static_assert(kPoolTileBlocks * kPoolBlock == kTileKeys, "a tile is 16 pool blocks");

// Shape of the decode (one query per group) configuration.
#ifndef CSA_INDEX_DECODE_STAGES
#define CSA_INDEX_DECODE_STAGES 4
#endif
#ifndef CSA_INDEX_DECODE_GROUPS
#define CSA_INDEX_DECODE_GROUPS 2
#endif
#ifndef CSA_INDEX_DECODE_CTAS_PER_SM
#define CSA_INDEX_DECODE_CTAS_PER_SM 2
#endif
#ifndef CSA_INDEX_DECODE_STAGES_FP4
#define CSA_INDEX_DECODE_STAGES_FP4 8
#endif
// TMEM accumulators of the one-query configuration (E4M3, FP4)
#ifndef CSA_INDEX_DECODE_NBUF
#define CSA_INDEX_DECODE_NBUF 2
#endif
#ifndef CSA_INDEX_DECODE_NBUF_FP4
#define CSA_INDEX_DECODE_NBUF_FP4 2
#endif
// Shape of the Reindex (pool gather) configuration
#ifndef CSA_INDEX_POOL_STAGES
#define CSA_INDEX_POOL_STAGES 4
#endif
#ifndef CSA_INDEX_POOL_STAGES_FP4
#define CSA_INDEX_POOL_STAGES_FP4 8
#endif
#ifndef CSA_INDEX_POOL_GROUPS
#define CSA_INDEX_POOL_GROUPS 2
#endif
#ifndef CSA_INDEX_POOL_CTAS_PER_SM
#define CSA_INDEX_POOL_CTAS_PER_SM 2
#endif
#ifndef CSA_INDEX_POOL_NBUF
#define CSA_INDEX_POOL_NBUF 2
#endif

// Kernel variants (template bits): the Reindex layer's pool gathers, the
// Full layer's block maxima, bf16 score stores, FP4 keys and queries.  Each
// launch runs the one variant it needs, so the decode kernel carries none of
// the others.
constexpr int kModePool = 1, kModeBlocks = 2, kModeBf16 = 4, kModeFp4 = 8;

template <int QPC, int kMode>
struct IndexCfg {
  static constexpr bool kFp4 = (kMode & kModeFp4) != 0, kPool = (kMode & kModePool) != 0;
  static constexpr int N = kIdxHeads * QPC;
  // Epilogue groups of 4 warps (one per TMEM lane quadrant).  One query per
  // group: the groups take tiles in turn; more queries: a group per query.
  static constexpr int GROUPS = QPC != 1 ? QPC : (kPool ? CSA_INDEX_POOL_GROUPS : CSA_INDEX_DECODE_GROUPS);
  static constexpr int EPI_WARPS = 4 * GROUPS;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int CTAS_PER_SM =
      QPC != 1 ? 1 : (kPool ? CSA_INDEX_POOL_CTAS_PER_SM : CSA_INDEX_DECODE_CTAS_PER_SM);
  static constexpr int STAGES =
      QPC != 1 ? (kFp4 ? 16 : 8)
               : kPool ? (kFp4 ? CSA_INDEX_POOL_STAGES_FP4 : CSA_INDEX_POOL_STAGES)
                       : (kFp4 ? CSA_INDEX_DECODE_STAGES_FP4 : CSA_INDEX_DECODE_STAGES);
  // TMEM accumulators; tile n uses accumulator n % NBUF
  static constexpr int NBUF = QPC != 1 ? 2
                              : kPool  ? CSA_INDEX_POOL_NBUF
                                       : (kFp4 ? CSA_INDEX_DECODE_NBUF_FP4 : CSA_INDEX_DECODE_NBUF);
  static_assert(QPC != 1 || NBUF >= GROUPS, "every epilogue group owns an accumulator");
  // Operand rows: 128 E4M3 bytes, or 64 bytes of E2M1 codes (plus scales).
  static constexpr uint32_t ROW = kFp4 ? kIdxDim / 2 : kIdxDim;
  static constexpr uint32_t KEY_TILE = kTileKeys * ROW;  // 16 or 8 KiB
  static constexpr uint32_t QBYTES = kIdxHeads * ROW;    // 8 or 4 KiB per query
  static constexpr uint32_t SF = kFp4 ? kSfBytes : 0;
  // TMEM columns: NBUF accumulators of N; FP4: 4 scale columns per
  // accumulator (the key tile's atom) and per query of either q^I buffer.
  static constexpr uint32_t SFA_COL = NBUF * N;
  static constexpr uint32_t SFB_COL = SFA_COL + 4 * NBUF;
  static constexpr uint32_t COLS = kFp4 ? SFB_COL + 4 * 2 * QPC : NBUF * N;
  static_assert(COLS <= 512, "TMEM holds 512 columns");
  static constexpr uint32_t TMEM_COLS =
      COLS <= 32 ? 32 : (COLS <= 64 ? 64 : (COLS <= 128 ? 128 : (COLS <= 256 ? 256 : 512)));
  static_assert(TMEM_COLS * CTAS_PER_SM <= 512, "the resident CTAs' accumulators share an SM's TMEM");
  // one query per CTA: each epilogue group gathers the row's first-digit
  // counts in shared memory and adds them to the global row once per query
  // group
  static constexpr uint32_t HIST = QPC == 1 ? GROUPS * kKeyBins * 4 : 0;
  static constexpr size_t SMEM = 1024 + 2 * QPC * (QBYTES + SF) + STAGES * (KEY_TILE + SF) + HIST +
                                 EPI_WARPS * kIdxHeads * 4 + (2 * STAGES + 2 * NBUF + 5) * 8 + 16;
};

// Work split: the flattened (query group, key tile) space is cut into
// gridDim.x equal contiguous ranges, one per CTA, with gridDim.x a multiple of
// the CTAs an SM holds; a range may cross into the next query group, whose
// q^I is then loaded into the other of two q^I buffers.  Tiles past a group's
// last visible key are skipped by every role alike.
struct GroupInfo {
  int64_t vis[4];   // visible entries (pool mode: pool slots to score) of each query of the group
  int64_t vent[4];  // visible entries of each query of the group
  int64_t vmax;
  int b, q0;
};

template <int QPC>
__device__ __forceinline__ GroupInfo group_info(const IndexArgs& a, int64_t g, int groups_per_seq) {
  GroupInfo gi;
  gi.b = static_cast<int>(g / groups_per_seq);
  gi.q0 = static_cast<int>(g % groups_per_seq) * QPC;
  gi.vmax = 0;
#pragma unroll
  for (int j = 0; j < QPC; ++j) {
    const int q = gi.q0 + j;
    int64_t V = 0;
    if (q < a.Q) {
      const int64_t t = a.q_pos ? static_cast<int64_t>(__ldg(a.q_pos + static_cast<int64_t>(gi.b) * a.Q + q))
                                : a.pos_base + q;
      V = t >= 0 ? (t + 1) / a.m : 0;
      if (V > a.n_cap) V = a.n_cap;
    }
    gi.vent[j] = V;
    if (a.pool) {  // the pool holds min(pool_blocks, ceil(V/8)) blocks
      const int64_t nb = (V + kPoolBlock - 1) / kPoolBlock;
      V = (nb < a.pool_blocks ? nb : a.pool_blocks) * kPoolBlock;
    }
    gi.vis[j] = V;
    gi.vmax = V > gi.vmax ? V : gi.vmax;
  }
  return gi;
}

// A score into its row: fp32, or its bf16 bits (already rounded).
template <bool kBf16>
__device__ __forceinline__ void store_score(uint8_t* row, int64_t i, float v) {
  if constexpr (kBf16)
    reinterpret_cast<uint16_t*>(row)[i] = static_cast<uint16_t>(__float_as_uint(v) >> 16);
  else
    reinterpret_cast<float*>(row)[i] = v;
}

// True if a query of the group sits past what the cache holds (V(t) > n_cap).
template <int QPC>
__device__ __forceinline__ bool group_past_cache(const IndexArgs& a, const GroupInfo& gi) {
  bool past = false;
#pragma unroll
  for (int j = 0; j < QPC; ++j) {
    const int q = gi.q0 + j;
    if (q < a.Q) {
      const int64_t t = a.q_pos ? static_cast<int64_t>(__ldg(a.q_pos + static_cast<int64_t>(gi.b) * a.Q + q))
                                : a.pos_base + q;
      past |= t >= 0 && (t + 1) / a.m > a.n_cap;
    }
  }
  return past;
}

template <int QPC, int kMode>
__global__ void __launch_bounds__(IndexCfg<QPC, kMode>::THREADS, IndexCfg<QPC, kMode>::CTAS_PER_SM)
    index_score_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                       const IndexArgs a, const int tiles_per_group, const int groups_per_seq) {
  constexpr bool kPool = (kMode & kModePool) != 0, kBlocks = (kMode & kModeBlocks) != 0,
                 kBf16 = (kMode & kModeBf16) != 0, kFp4 = (kMode & kModeFp4) != 0;
  using Cfg = IndexCfg<QPC, kMode>;
  constexpr int N = Cfg::N;
  constexpr int STAGES = Cfg::STAGES;
  constexpr uint32_t kKeyTileBytes = Cfg::KEY_TILE, kQBytes = Cfg::QBYTES;
  pdl_launch_dependents();
  // Without a.early: wait before any global access and before TMEM is
  // taken.  With it the predecessor is the counters' zeroing kernel, whose
  // own predecessor has completed (no other kernel of the stream holds TMEM
  // or writes this launch's inputs): the producer streams key tiles before
  // the wait, up to each query's last visible tile, and the epilogue waits
  // before its first global access (the counters the zeroing kernel clears).
  const bool early = !kPool && a.early != 0;
  if (!early) pdl_wait();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = base;                                   // [2][QPC][QBYTES]
  uint8_t* k_s = q_s + 2 * QPC * kQBytes;                // [STAGES][KEY_TILE]
  uint8_t* ksf_s = k_s + STAGES * kKeyTileBytes;         // FP4: [STAGES][512] scale atoms
  uint8_t* qsf_s = ksf_s + STAGES * Cfg::SF;             // FP4: [2][QPC][512] query scale records
  constexpr int NBUF = Cfg::NBUF;
  constexpr int kEpiWarps = Cfg::EPI_WARPS;
  constexpr int kEpiGroups = Cfg::GROUPS;
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(qsf_s + 2 * QPC * Cfg::SF);  // QPC 1: [GROUPS][2048] digit counts
  float* w_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(hist_s) + Cfg::HIST);  // [epilogue warps][64]
  uint64_t* full = reinterpret_cast<uint64_t*>(w_s + kEpiWarps * kIdxHeads);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [NBUF]
  uint64_t* acc_empty = acc_full + NBUF; // [NBUF]
  uint64_t* q_full = acc_empty + NBUF;   // [2]
  uint64_t* q_empty = q_full + 2;     // [2]
  uint64_t* mma_done = q_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n_groups = static_cast<int64_t>(a.B) * groups_per_seq;
  const int64_t units = n_groups * tiles_per_group;
  const int64_t u0 = units * blockIdx.x / gridDim.x;
  const int64_t u1 = units * (blockIdx.x + 1) / gridDim.x;
  if (u0 >= u1) return;

  if (warp == 1) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int x = 0; x < NBUF; ++x) {
      mbar_init(&acc_full[x], 1);
      // one query per tile: the owning group's 4 warps; else every epilogue warp
      mbar_init(&acc_empty[x], QPC == 1 ? 4 : kEpiWarps);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_empty[x], 1);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  static_assert(!kPool || QPC == 1, "a pool belongs to one query");
  if (kPool && warp == 0) {
    // ---------------- TMA producer, Reindex layer (whole warp) ----------------
    // A tile is 16 pool blocks of 8 keys; lane l < 16 loads slot l's block
    // into its 1 KiB swizzle atom with its own TMA box.  Unit u's block ids
    // are pool[16u .. 16u+15] (one query per group, pool_ld == pool_blocks);
    // every lane keeps its slot's ids for the next kAhead units in flight.
    // A slot without a block, or with an id outside the cache, loads block 0,
    // which the epilogue does not score.
    // FP4: the tile's scale atom is assembled here.  Block blk's 8 scale
    // words lie on lines 8*(blk%4) .. +7, word (blk%16)/4, of the sequence's
    // atom blk/16; slot l's go to lines 8*(l%4) .. +7, word l/4 of the
    // stage's atom.  Lane l loads them kAhead units ahead (its ids are read
    // 2*kAhead units ahead), stores them when the stage is free and fences
    // them for the tensor cores before lane 0 arrives on the stage.
    constexpr int kAhead = 4;
    constexpr int kIdAhead = kFp4 ? 2 * kAhead : kAhead;
    const int64_t n_blk = (a.n_cap + kPoolBlock - 1) / kPoolBlock;
    const int32_t* ids = a.pool + (lane & (kPoolTileBlocks - 1));
    int32_t ring[kIdAhead];
#pragma unroll
    for (int d = 0; d < kIdAhead; ++d) ring[d] = u0 + d < u1 ? __ldg(ids + kPoolTileBlocks * (u0 + d)) : 0;
    uint32_t sw[kFp4 ? kAhead : 1][8];
    const auto load_scales = [&](int64_t up, int32_t id, uint32_t(&w)[8]) {
      const bool live = lane < kPoolTileBlocks && up < u1;
      const int32_t blk = (id >= 0 && id < n_blk) ? id : 0;
      const int64_t bp = live ? up / tiles_per_group / groups_per_seq : 0;
      const uint8_t* src = a.kI_sf + bp * a.kI_sf_ld + (blk >> 4) * static_cast<int64_t>(kSfBytes) + (blk & 3) * 128 +
                           ((blk & 15) >> 2) * 4;
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = live ? __ldg(reinterpret_cast<const uint32_t*>(src + 16 * k)) : 0u;
    };
    if constexpr (kFp4) {
#pragma unroll
      for (int d = 0; d < kAhead; ++d) load_scales(u0 + d, ring[d], sw[d]);
    }
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_q);
    }
    const uint64_t pol = policy_evict_first();
    uint32_t issued = 0, parity = 0;
    uint32_t q_uses[2] = {0, 0};
    int64_t seen_g = -1;
    bool active = false;
    GroupInfo gi{};
    int qb = 1, it = 0;
    bool ok = true;
    int64_t g = u0 / tiles_per_group, tile = u0 % tiles_per_group - 1;
    for (int64_t u = u0; u < u1 && ok; ++u) {
      const int32_t id = ring[0];
#pragma unroll
      for (int d = 0; d + 1 < kIdAhead; ++d) ring[d] = ring[d + 1];
      ring[kIdAhead - 1] = u + kIdAhead < u1 ? __ldg(ids + kPoolTileBlocks * (u + kIdAhead)) : 0;
      uint32_t cur[8];
      if constexpr (kFp4) {  // this unit's scale words; load those of unit u + kAhead
#pragma unroll
        for (int k = 0; k < 8; ++k) cur[k] = sw[0][k];
#pragma unroll
        for (int d = 0; d + 1 < kAhead; ++d)
#pragma unroll
          for (int k = 0; k < 8; ++k) sw[d][k] = sw[d + 1][k];
        load_scales(u + kAhead, ring[kAhead - 1], sw[kAhead - 1]);
      }
      if (++tile == tiles_per_group) {
        tile = 0;
        ++g;
      }
      if (g != seen_g) {
        gi = group_info<QPC>(a, g, groups_per_seq);
        seen_g = g;
        active = gi.vmax > tile * kTileKeys;
        if (active) {
          qb ^= 1;
          if (lane == 0) {
            if (q_uses[qb] > 0) ok = mbar_wait(&q_empty[qb], (q_uses[qb] - 1) & 1u, a.status);
            if (ok) {
              const int64_t r = static_cast<int64_t>(gi.b) * a.Q + gi.q0;
              mbar_arrive_expect_tx(&q_full[qb], kQBytes + Cfg::SF);
              tma_load_2d(q_s + qb * kQBytes, &tm_q, 0, static_cast<int32_t>(r * kIdxHeads), &q_full[qb]);
              if constexpr (kFp4) bulk_load(qsf_s + qb * kSfBytes, a.qI_sf + r * kSfBytes, kSfBytes, &q_full[qb]);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          ++q_uses[qb];
        }
      }
      if (!active || tile * kTileKeys >= gi.vmax) continue;
      const int st = it % STAGES;
      const uint32_t use = static_cast<uint32_t>(it / STAGES);
      if (lane == 0 && use > 0) ok = mbar_wait(&empty[st], (use - 1) & 1u, a.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if constexpr (kFp4) {
        if (lane < kPoolTileBlocks) {
          uint8_t* dst = ksf_s + st * kSfBytes + (lane & 3) * 128 + (lane >> 2) * 4;
#pragma unroll
          for (int k = 0; k < 8; ++k) *reinterpret_cast<uint32_t*>(dst + 16 * k) = cur[k];
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (it == 0 && test_fault(a.status, kFaultIndexer)) {  // test fault: the first tile is never loaded (the MMA's wait gives up)
        ++it;
        continue;
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[st], kKeyTileBytes);
      if (lane < kPoolTileBlocks) {
        const int32_t blk = (id >= 0 && id < n_blk) ? id : 0;
        tma_load_3d(k_s + st * kKeyTileBytes + lane * (kPoolBlock * Cfg::ROW), &tm_k, 0, blk * kPoolBlock, gi.b,
                    &full[st], pol);
      }
      issued |= 1u << st;
      parity = (parity & ~(1u << st)) | ((use & 1u) << st);
      ++it;
    }
    // Our own copies must have landed before the CTA may exit.
    if (lane == 0) {
      for (int x = 0; x < STAGES; ++x)
        if (issued & (1u << x)) mbar_wait(&full[x], (parity >> x) & 1u, a.status);
      for (int x = 0; x < 2; ++x)
        if (q_uses[x]) mbar_wait(&q_full[x], (q_uses[x] - 1) & 1u, a.status);
    }
    __syncwarp();
  } else if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_q);
      const uint64_t pol = policy_evict_first();
      uint32_t issued = 0, parity = 0;
      uint32_t q_uses[2] = {0, 0};
      int64_t seen_g = -1;
      bool active = false;
      GroupInfo gi{};
      int qb = 1, it = 0;
      bool ok = true, waited = false;
      int64_t g = u0 / tiles_per_group, tile = u0 % tiles_per_group - 1;
      for (int64_t u = u0; u < u1 && ok; ++u) {
        if (++tile == tiles_per_group) {  // advance (group, tile) without dividing
          tile = 0;
          ++g;
        }
        if (g != seen_g) {
          gi = group_info<QPC>(a, g, groups_per_seq);
          seen_g = g;
          active = gi.vmax > tile * kTileKeys;  // the group has work in this range
          if (active) {
            qb ^= 1;
            if (q_uses[qb] > 0 && !(ok = mbar_wait(&q_empty[qb], (q_uses[qb] - 1) & 1u, a.status))) break;
            mbar_arrive_expect_tx(&q_full[qb], QPC * (kQBytes + Cfg::SF));
            for (int j = 0; j < QPC; ++j) {
              const int64_t r = static_cast<int64_t>(gi.b) * a.Q + gi.q0 + j;
              tma_load_2d(q_s + (qb * QPC + j) * kQBytes, &tm_q, 0, static_cast<int32_t>(r * kIdxHeads),
                          &q_full[qb]);
              if constexpr (kFp4) {  // a query past the last one reads the last record (not scored)
                const int64_t rc = r < static_cast<int64_t>(a.B) * a.Q ? r : static_cast<int64_t>(a.B) * a.Q - 1;
                bulk_load(qsf_s + (qb * QPC + j) * kSfBytes, a.qI_sf + rc * kSfBytes, kSfBytes, &q_full[qb]);
              }
            }
            ++q_uses[qb];
          }
        }
        if (!active || tile * kTileKeys >= gi.vmax) continue;
        if (early && !waited && (tile + 1) * kTileKeys >= gi.vmax) {  // the tile may hold the new entry
          pdl_wait();
          waited = true;
        }
        const int s = it % STAGES;
        const uint32_t use = static_cast<uint32_t>(it / STAGES);
        if (use > 0 && !(ok = mbar_wait(&empty[s], (use - 1) & 1u, a.status))) break;
        if (it == 0 && test_fault(a.status, kFaultIndexer)) {  // test fault: the first tile is never loaded (the MMA's wait gives up)
          ++it;
          continue;
        }
        mbar_arrive_expect_tx(&full[s], kKeyTileBytes + Cfg::SF);
        tma_load_3d(k_s + s * kKeyTileBytes, &tm_k, 0, static_cast<int32_t>(tile * kTileKeys), gi.b, &full[s], pol);
        if constexpr (kFp4)
          bulk_load(ksf_s + s * kSfBytes, a.kI_sf + static_cast<int64_t>(gi.b) * a.kI_sf_ld + tile * kSfBytes, kSfBytes,
                    &full[s], pol);
        issued |= 1u << s;
        parity = (parity & ~(1u << s)) | ((use & 1u) << s);
        ++it;
      }
      // Our own copies must have landed before the CTA may exit.
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) mbar_wait(&full[s], (parity >> s) & 1u, a.status);
      for (int x = 0; x < 2; ++x)
        if (q_uses[x]) mbar_wait(&q_full[x], (q_uses[x] - 1) & 1u, a.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(kTileKeys, N, 0, 0, 0, 0);
      // FP4: the scale atoms go to TMEM by tcgen05.cp, source described as
      // 32 contiguous 16-byte lines
      const auto sf_desc = [](const uint8_t* p) { return smem_desc(smem_u32(p), 128, 128, kSwizzleNone); };
      uint32_t q_uses[2] = {0, 0};
      int64_t seen_g = -1;
      bool active = false;
      GroupInfo gi{};
      int qb = 1, it = 0;
      bool ok = true;
      int64_t g = u0 / tiles_per_group, tile = u0 % tiles_per_group - 1;
      for (int64_t u = u0; u < u1 && ok; ++u) {
        if (++tile == tiles_per_group) {  // advance (group, tile) without dividing
          tile = 0;
          ++g;
        }
        if (g != seen_g) {
          gi = group_info<QPC>(a, g, groups_per_seq);
          seen_g = g;
          active = gi.vmax > tile * kTileKeys;
          if (active) {
            if (q_uses[qb] > 0) tc_commit(&q_empty[qb]);  // previous group's buffer is free once its MMAs end
            qb ^= 1;
            if (!(ok = mbar_wait(&q_full[qb], q_uses[qb] & 1u, a.status))) break;
            ++q_uses[qb];
            if constexpr (kFp4) {
              tc_fence_after();
              for (int j = 0; j < QPC; ++j)
                tc_cp_32x128b_warpx4(tmem + Cfg::SFB_COL + 4 * (qb * QPC + j), sf_desc(qsf_s + (qb * QPC + j) * kSfBytes));
            }
          }
        }
        if (!active || tile * kTileKeys >= gi.vmax) continue;
        const int s = it % STAGES;
        const uint32_t use = static_cast<uint32_t>(it / STAGES);
        const int x = it % NBUF;
        const uint32_t xuse = static_cast<uint32_t>(it / NBUF);
        if (xuse > 0 && !(ok = mbar_wait(&acc_empty[x], (xuse - 1) & 1u, a.status))) break;
        if (!(ok = mbar_wait(&full[s], use & 1u, a.status))) break;
        tc_fence_after();
        const uint32_t kb = smem_u32(k_s + s * kKeyTileBytes);
        const uint32_t qbase = smem_u32(q_s + qb * QPC * kQBytes);
        if constexpr (kFp4) {
          // K = 128 as two block-scaled MMAs of 64 (scale bytes 0-1, then
          // 2-3); one MMA per query, each with its own scale columns
          const uint32_t sfa = tmem + Cfg::SFA_COL + 4 * x;
          tc_cp_32x128b_warpx4(sfa, sf_desc(ksf_s + s * kSfBytes));
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t ad = smem_desc(kb + kk * 32, 16, 512, kSwizzle64B);
#pragma unroll
            for (int j = 0; j < QPC; ++j) {
              const uint64_t bd = smem_desc(qbase + j * kQBytes + kk * 32, 16, 512, kSwizzle64B);
              mma_mxf4(tmem + x * N + j * kIdxHeads, ad, bd, instr_desc_mxf4(kTileKeys, kIdxHeads, 2 * kk, 2 * kk),
                       sfa, tmem + Cfg::SFB_COL + 4 * (qb * QPC + j), kk > 0 ? 1u : 0u);
            }
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < kIdxDim / 32; ++kk) {
            const uint64_t ad = smem_desc(kb + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(qbase + kk * 32, 16, 1024, kSwizzle128B);
            mma_f8(tmem + x * N, ad, bd, idesc, kk > 0 ? 1u : 0u);
          }
        }
        tc_commit(&empty[s]);
        tc_commit(&acc_full[x]);
        ++it;
      }
      tc_commit(mma_done);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue ----------------
    // Groups of 4 warps; in a group, warp w reads TMEM lane quadrant w % 4
    // (keys 32*(w%4) .. +31 of the tile).  With one query per tile the groups
    // take tiles in turn; with more, every group takes every tile and scores
    // its own query.
    // The CTA's unit range is walked group by group: a group's active tiles
    // are the prefix of its tiles below its last visible key, so the running
    // tile count `it` (the MMA thread's accumulator numbering) advances by a
    // group's active tiles at once, and a warp visits only its own tiles.
    if (early) pdl_wait();
    const int ew = warp - 2;
    const int grp = ew >> 2;
    const int sub = warp & 3;
    const int row = sub * 32 + lane;
    const int jq = QPC == 1 ? 0 : grp;  // the query this group scores
    float* w_mine = w_s + ew * kIdxHeads;  // this warp's copy of the head weights
    const uint32_t w_addr = smem_u32(w_mine);
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(sub * 32) << 16) + jq * kIdxHeads;
    constexpr int kStep = QPC == 1 ? kEpiGroups : 1;
    // One query per CTA, many CTAs per row (a.hist_private): each epilogue
    // group counts digits in its own hist_s row and adds it to the global
    // row once it is done with the query group, instead of many CTAs'
    // atomics meeting on the same bins.  The group's 4 warps meet at named
    // barrier 1 + grp around each flush; a warp whose wait gave up still
    // walks the groups (doing no work) so that no barrier hangs.
    const bool priv = QPC == 1 && a.hist_private && a.hist;
    const uint32_t et = threadIdx.x - 64 - 128 * grp;  // thread index within the epilogue group
    uint32_t* hist_mine = hist_s + grp * kKeyBins;
    if (priv) {
      for (uint32_t i = et; i < kKeyBins; i += 128) hist_mine[i] = 0u;
      named_bar_sync(1 + grp, 128);
    }
    int it = 0;
    bool ok = true;
    for (int64_t g = u0 / tiles_per_group; g * tiles_per_group < u1; ++g) {
      const int64_t gu = g * tiles_per_group;
      const int ta = gu < u0 ? static_cast<int>(u0 - gu) : 0;
      const int te = u1 - gu < tiles_per_group ? static_cast<int>(u1 - gu) : tiles_per_group;
      const GroupInfo gi = group_info<QPC>(a, g, groups_per_seq);
      const int64_t n_vis_tiles = (gi.vmax + kTileKeys - 1) / kTileKeys;
      const int tb = n_vis_tiles < te ? static_cast<int>(n_vis_tiles) : te;
      if (tb <= ta) continue;
      if (ta == 0 && warp == 2 && lane == 0 && group_past_cache<QPC>(a, gi)) record_error(a.status, kErrIndexRange);
      // this group's query: head weights, output rows, visible counts
      const int q = gi.q0 + jq;
      const int64_t row_off = static_cast<int64_t>(gi.b) * a.Q + q;
      __syncwarp();  // the warp is done with the previous group's weights
      for (int e = lane; e < kIdxHeads; e += 32) {
        const uint16_t wb = q < a.Q ? a.wI[row_off * kIdxHeads + e] : uint16_t(0);
        w_mine[e] = __uint_as_float(static_cast<uint32_t>(wb) << 16);
      }
      __syncwarp();
      const int64_t vis = gi.vis[jq], vent = gi.vent[jq];
      uint8_t* srow = reinterpret_cast<uint8_t*>(a.scores) + row_off * a.score_ld * (kBf16 ? 2 : 4);
      uint32_t* hrow = a.hist ? a.hist + row_off * kKeyBins : nullptr;
      const int32_t* prow = kPool ? a.pool + row_off * a.pool_ld : nullptr;
      const int64_t n_blk_vis = (vent + kPoolBlock - 1) / kPoolBlock;
      int t = ta;
      if constexpr (kStep > 1) t += ((grp - it) % kStep + kStep) % kStep;
      for (; ok && t < tb; t += kStep) {
        const int my_it = it + (t - ta);
        const int x = my_it % NBUF;
        const uint32_t xuse = static_cast<uint32_t>(my_it / NBUF);
        // every lane waits; the warp leaves together if any lane gave up
        if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[x], xuse & 1u, a.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int64_t s_idx = static_cast<int64_t>(t) * kTileKeys + row;
        const uint32_t taddr = t_lane + x * N;
        // four independent chains (head h into chain h % 4), two to a packed
        // register: each step is fmaf(w_h, fmaxf(s_h, 0), chain) per head
        // (measured faster than the same math through the packed-FMA
        // intrinsics with separate weight loads)
        uint64_t acc01 = 0ull, acc23 = 0ull;
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // 32 heads at a time keeps registers low
          uint32_t r[32];
          tmem_ld32(taddr + 32 * half, r);
          tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            relu_fma4(acc01, acc23, w_addr + 16 * (8 * half + v), r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
        }
        const float acc[4] = {__uint_as_float(static_cast<uint32_t>(acc01)), __uint_as_float(static_cast<uint32_t>(acc01 >> 32)),
                              __uint_as_float(static_cast<uint32_t>(acc23)), __uint_as_float(static_cast<uint32_t>(acc23 >> 32))};
        float score = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        // bf16 scores: every use below (store, digit counts, block maxima)
        // sees the rounded value
        if constexpr (kBf16) score = __bfloat162float(__float2bfloat16_rn(score));
        const bool in_row = s_idx < vis;
        bool valid = in_row;
        if (kPool && in_row) {  // slot s_idx holds entry 8*pool[s_idx/8] + s_idx%8
          const int32_t blk = __ldg(prow + (s_idx >> 3));
          if (blk >= n_blk_vis && (row & 7) == 0) record_error(a.status, kErrIndexRange);
          valid = blk >= 0 && static_cast<int64_t>(blk) * kPoolBlock + (row & 7) < vent;
          store_score<kBf16>(srow, s_idx, valid ? score : -INFINITY);
        } else if (valid) {
          store_score<kBf16>(srow, s_idx, score);
        }
        if constexpr (kBlocks) {  // the block's largest score: 8 adjacent lanes
          float bm = valid ? score : -INFINITY;
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
          const bool lead = valid && (lane & 7) == 0;  // the block's first entry is visible
          if (lead) a.block_scores[row_off * a.block_ld + (s_idx >> 3)] = bm;
          const int bbin = lead ? static_cast<int>(score_key(bm) >> kKeyBinShift) : -1;
          const unsigned bpeers = __match_any_sync(0xffffffffu, bbin);
          if (lead && lane == __ffs(bpeers) - 1) atomicAdd(a.block_hist + row_off * kKeyBins + bbin, __popc(bpeers));
        }
        if (hrow) {  // first-digit histogram of the row, one atomic per distinct digit per warp
          const int bin = valid ? static_cast<int>(score_key(score) >> kKeyBinShift) : -1;
          const unsigned peers = __match_any_sync(0xffffffffu, bin);
          if (valid && lane == __ffs(peers) - 1) {
            if (priv)
              atomicAdd(hist_mine + bin, __popc(peers));  // shared
            else
              atomicAdd(hrow + bin, __popc(peers));  // global
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[x]);
      }
      it += tb - ta;
      if (priv) {  // this group is done with the query: add its counts to the row
        named_bar_sync(1 + grp, 128);
        for (uint32_t i = et; i < kKeyBins; i += 128) {
          const uint32_t c = hist_mine[i];
          if (c) {
            atomicAdd(hrow + i, c);
            hist_mine[i] = 0u;
          }
        }
        named_bar_sync(1 + grp, 128);
      }
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) mbar_wait(mma_done, 0, a.status);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

bool encode_maps(const IndexArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* tm_k,
                 CUtensorMap* tm_q) {
  // Rows of 128 E4M3 bytes (128-byte swizzle) or of 64 bytes of E2M1 codes
  // (64-byte swizzle).
  const cuuint64_t row = a.fp4 ? kIdxDim / 2 : kIdxDim;
  const CUtensorMapSwizzle swz = a.fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  // K^I: [B][n_cap][row] bytes, box = 128 keys of one sequence (pool mode:
  // one block of 8 keys).
  cuuint64_t kdim[3] = {row, static_cast<cuuint64_t>(a.n_cap), static_cast<cuuint64_t>(a.B)};
  cuuint64_t kstride[2] = {row, static_cast<cuuint64_t>(a.n_cap) * row};
  cuuint32_t kbox[3] = {static_cast<cuuint32_t>(row), static_cast<cuuint32_t>(a.pool ? kPoolBlock : kTileKeys), 1};
  cuuint32_t ones[3] = {1, 1, 1};
  if (encode(tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.kI), kdim, kstride, kbox, ones,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  // q^I: [B*Q*64 rows][row bytes], box = the 64 heads of one query.
  cuuint64_t qdim[2] = {row, static_cast<cuuint64_t>(a.B) * static_cast<cuuint64_t>(a.Q) * kIdxHeads};
  cuuint64_t qstride[1] = {row};
  cuuint32_t qbox[2] = {static_cast<cuuint32_t>(row), static_cast<cuuint32_t>(kIdxHeads)};
  return encode(tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.qI), qdim, qstride, qbox, ones,
                CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int QPC, int kMode>
cudaError_t launch_qpc(const IndexArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode, cudaStream_t stream) {
  using Cfg = IndexCfg<QPC, kMode>;
  CUtensorMap tm_k, tm_q;
  if (!encode_maps(a, encode, &tm_k, &tm_q)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(index_score_kernel<QPC, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg::SMEM));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_sm = Cfg::CTAS_PER_SM;
  const int64_t tiles_per_group =
      a.pool ? a.pool_blocks / kPoolTileBlocks : (a.n_cap + kTileKeys - 1) / kTileKeys;
  const int64_t groups_per_seq = (a.Q + QPC - 1) / QPC;
  const int64_t units = tiles_per_group * groups_per_seq * a.B;
  // One wave of CTAs that all stay resident; each takes an equal range.
  int64_t ctas = static_cast<int64_t>(sms) * per_sm;
  if (ctas > units) ctas = units;
  // shared-memory digit counts pay off when many CTAs share a row and each
  // has many tiles to count
  IndexArgs ka = a;
  const int64_t rows = static_cast<int64_t>(a.B) * a.Q;
  ka.hist_private = QPC == 1 && ctas >= 8 * rows && units >= 16 * ctas;
  return launch_pdl(index_score_kernel<QPC, kMode>, dim3(static_cast<unsigned>(ctas)), dim3(Cfg::THREADS), Cfg::SMEM,
                    stream, tm_k, tm_q, ka, static_cast<int>(tiles_per_group), static_cast<int>(groups_per_seq));
}

}  // namespace

cudaError_t launch_index_scores(const IndexArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode,
                                cudaStream_t stream) {
  if (a.B <= 0 || a.Q <= 0) return cudaSuccess;
  if (a.pool && (a.pool_blocks <= 0 || a.pool_blocks % kPoolTileBlocks != 0 || a.pool_ld != a.pool_blocks))
    return cudaErrorInvalidValue;
  const int mode = (a.pool ? kModePool : 0) | (a.block_scores ? kModeBlocks : 0) | (a.bf16_scores ? kModeBf16 : 0);
  if (a.fp4) {  // FP4 keys and queries: one query per CTA, or three (TMEM holds two accumulators of 3 x 64)
    if (!a.kI_sf || !a.qI_sf) return cudaErrorInvalidValue;
    constexpr int F = kModeFp4, L = kModeBlocks, H = kModeBf16, P = kModePool;
    if (a.Q >= 3 && !a.pool) {
      switch (mode) {
        case 0: return launch_qpc<3, F>(a, encode, stream);
        case L: return launch_qpc<3, F | L>(a, encode, stream);
        case H: return launch_qpc<3, F | H>(a, encode, stream);
        case L | H: return launch_qpc<3, F | L | H>(a, encode, stream);
        default: return cudaErrorInvalidValue;
      }
    }
    switch (mode) {
      case 0: return launch_qpc<1, F>(a, encode, stream);
      case L: return launch_qpc<1, F | L>(a, encode, stream);
      case H: return launch_qpc<1, F | H>(a, encode, stream);
      case L | H: return launch_qpc<1, F | L | H>(a, encode, stream);
      case P: return launch_qpc<1, F | P>(a, encode, stream);
      case P | H: return launch_qpc<1, F | P | H>(a, encode, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (a.Q >= 4 && !a.pool) {  // a pool is per query: one query per tile
    switch (mode) {
      case 0: return launch_qpc<4, 0>(a, encode, stream);
      case kModeBlocks: return launch_qpc<4, kModeBlocks>(a, encode, stream);
      case kModeBf16: return launch_qpc<4, kModeBf16>(a, encode, stream);
      case kModeBlocks | kModeBf16: return launch_qpc<4, kModeBlocks | kModeBf16>(a, encode, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (mode) {
    case 0: return launch_qpc<1, 0>(a, encode, stream);
    case kModePool: return launch_qpc<1, kModePool>(a, encode, stream);
    case kModeBlocks: return launch_qpc<1, kModeBlocks>(a, encode, stream);
    case kModeBf16: return launch_qpc<1, kModeBf16>(a, encode, stream);
    case kModePool | kModeBf16: return launch_qpc<1, kModePool | kModeBf16>(a, encode, stream);
    case kModeBlocks | kModeBf16: return launch_qpc<1, kModeBlocks | kModeBf16>(a, encode, stream);
    default: return cudaErrorInvalidValue;  // a pool with block outputs is not a call of this library
  }
}

}  // namespace csa
