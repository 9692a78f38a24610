// Host-side launchers of the CSA kernels (internal to libcsa; the public C ABI
// is include/csa.h).  Every launcher enqueues on `stream` and returns the
// launch's cudaError_t; arguments are validated by the C-ABI layer first.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

// Counts successful kernel launches (reported by csa_launch_count).
void note_launch();
inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) note_launch();
  return e;
}

// Launches a kernel with programmatic stream serialization (and, for
// cluster_x > 1, in clusters of cluster_x CTAs along x): it may start (and
// wait in pdl_wait) while the kernel before it in the stream finishes, which
// hides the launch gap between the stages.  Every kernel of this library
// calls pdl_launch_dependents() and then pdl_wait() before its first global
// memory access, so stream order holds for all data.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  return counted(cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...));
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  return launch_pdl_cluster(kernel, grid, block, smem, stream, 1u, static_cast<Args&&>(args)...);
}

// Fixed model dimensions the kernels are specialised for.
constexpr int kHeads = 64;      // query heads
constexpr int kDim = 512;       // shared K=V latent width
constexpr int kRope = 64;       // RoPE channels (the last kRope of kDim)
constexpr int kIdxHeads = 64;   // indexer heads
constexpr int kIdxDim = 128;    // indexer width (bytes of one e4m3 key row)
constexpr int kMaxTopk = 2048;
constexpr int kMaxWindow = 1024;
constexpr int kFp4Entry = kDim / 2 + kDim / 16;  // 288: E2M1 codes + one E4M3 scale per 16 values
constexpr int kPoolBlock = 8;         // entries per block of the hierarchical indexer's pool
constexpr int kPoolTileBlocks = 16;   // pool blocks per 128-key indexer tile

// RoPE angles as fixed-point fractions of a turn.  Frequency j of the
// partial RoPE, theta^(-2j/R), is held as f_j / (2 pi) * 2^64 (fp64 on the
// host, so its relative error is about 2^-52); the angle of an integer
// position p is then p * f_j / (2 pi) turns, whose fractional part is the
// low 64 bits of the integer product p * table[j] (a negative p wraps the
// same way).  Exact integer arithmetic on the device: no angle needs fp64 or
// a reduction modulo 2 pi; the angle, in [-pi, pi), goes to the hardware
// sine and cosine (absolute error about 5e-7 there), and the error at
// position 2^31 stays near 1e-6 rad in all.
void fill_rope_turns(double theta, uint64_t (&table)[kRope / 2]);
// sin and cos of position p's angle at the frequency whose table entry is turns.
__device__ __forceinline__ void rope_sincos(int64_t p, uint64_t turns, float* s, float* c) {
  const uint64_t frac = static_cast<uint64_t>(p) * turns;  // the angle modulo one turn, in 2^-64 turns
  const int32_t half = static_cast<int32_t>(frac >> 32);    // in half-turns times 2^31, in [-2^31, 2^31)
  __sincosf(static_cast<float>(half) * 1.4629180792671596e-09f, s, c);  // pi * 2^-31
}

// ---- compressor --------------------------------------------------------------
struct CompressArgs {
  int mode;                 // 0: bulk chunk, 1: decode ring (one entry at most)
  int B, m;
  int64_t n_new, entry0;    // bulk: entries entry0 .. entry0+n_new-1
  const uint16_t *Ca, *Za, *Cb, *Zb;  // bulk [B][m*n_new][D]; ring [B][2m][D]
  const uint16_t *Cb_prev, *Zb_prev;  // bulk [B][m][D] or null
  const uint16_t *Ba, *Bb, *rms_w;
  uint16_t* kv_out;
  int64_t kv_stride_b;      // elements between sequences of kv_out
  int64_t n_cap;            // ring mode: entries the cache holds
  const int32_t* q_pos;     // ring mode: [B] positions
  double rope_theta;
  float rms_eps;
  unsigned* status;
  uint64_t rope_turns[kRope / 2];  // theta^(-2j/R) / (2 pi) * 2^64 (fill_rope_turns), by launch_compress
  uint8_t* key_out;            // indexer keys (launch_index_keys): E4M3 rows of kIdxDim
  float* state;                // single-stream step: [B][3][kDim] running (max, sum, weighted sum)
  uint8_t* kv_fp4_out;         // main compressor: entries in the FP4 layout instead of kv_out
  int64_t fp4_stride_b;        // bytes between sequences of kv_fp4_out
};
// keys: optional bulk-mode arguments of the indexer's key compressor for
// the same entries (same B, m, n_new, entry0): warp 0 of each CTA writes the
// entry's indexer key too.
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t stream, const CompressArgs* keys = nullptr);
// The non-overlapped (single-stream) compressor, block size a.m (1..128):
// mode 0 bulk over Ca / Za (the stream's C / Z rows) with the optional slot
// bias Ba; mode 1 one decode token per sequence, Ca / Za [B][kDim], folded
// into a.state and finished into kv_out when it closes a block.
constexpr int kMaxSingleM = 128;
cudaError_t launch_compress_single(const CompressArgs& a, cudaStream_t stream);
// Indexer keys from 128-wide compressor rows (bulk mode): the compressor's
// steps at width kIdxDim, the Hadamard rotation, E4M3 codes into key_out.
cudaError_t launch_index_keys(const CompressArgs& a, cudaStream_t stream);

// ---- lightning indexer scores (tcgen05, FP8) -------------------------------------
struct IndexArgs {
  const uint8_t* qI;        // [B][Q][64][128] E4M3; FP4: [B][Q][64][64] E2M1 codes
  const uint16_t* wI;       // [B][Q][64]
  const uint8_t* kI;        // [B][n_cap][128] E4M3; FP4: [B][n_cap][64] E2M1 codes
  // FP4 indexer (CSA2): E8M0 scales of 32 channels.  Keys: per sequence, one
  // 512-byte atom per 128 entries (entry e at byte 16*(e%32) + 4*((e%128)/32)
  // + block of atom e/128); queries: one 512-byte record per query (head h at
  // byte 16*(h%32) + 4*(h/32) + block, bytes 8..15 of each line unused).
  int fp4;
  const uint8_t* kI_sf;     // [B][kI_sf_ld]
  int64_t kI_sf_ld;         // bytes between sequences: 512 * ceil(n_cap / 128)
  const uint8_t* qI_sf;     // [B*Q][512]
  const int32_t* q_pos;     // [B][Q] or null (then pos_base + q)
  int64_t pos_base;
  int B, Q, m;
  int64_t n_cap;
  float* scores;            // [B*Q][score_ld] fp32, or bf16 (uint16) with bf16_scores
  int64_t score_ld;         // elements (a multiple of 8)
  int bf16_scores;          // 1: scores rounded to bf16 and stored as 2 bytes
  uint32_t* hist;           // [B*Q][2048] key top-digit counts (zeroed by the caller) or null
  int hist_private;         // set by the launcher: count in shared memory, add to hist per query group
  // Full layer of the hierarchical indexer: per row, the largest score of
  // each block of kPoolBlock entries with a visible first entry, and the
  // first-digit counts of those block scores (zeroed by the caller).
  float* block_scores;      // [B*Q][block_ld] or null
  int64_t block_ld;
  uint32_t* block_hist;     // [B*Q][2048] or null
  // Reindex layer: score only the entries of the row's pool blocks (ascending
  // block ids, -1 padded); scores are then indexed by pool slot (8*j + r is
  // entry 8*pool[j] + r), -inf for slots that hold no visible entry.
  const int32_t* pool;      // [B*Q][pool_ld] or null
  int pool_blocks;          // a multiple of kPoolTileBlocks
  int64_t pool_ld;          // a multiple of 4
  // 1: the launch directly follows a launch_zero kernel of the same stream
  // (which lets its dependents start only once its own predecessor has
  // completed), so the kernel may read its inputs before waiting for that
  // kernel: q_pos, q^I and every key tile but each query's last visible one
  // (which may hold the entry that kernel writes).  Not for pool mode.
  int early;
  unsigned* status;
};
cudaError_t launch_index_scores(const IndexArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode,
                                cudaStream_t stream);
// Zeroes `bytes` (a multiple of 4) at a 16-byte aligned device pointer, as a
// kernel on the programmatic-launch chain.
// A decode step's new rows, written into the caches by the step's first
// kernel (the counters' zeroing) so that they cost no launch of their own:
// the window row of position t = q_pos[b] into ring slot t mod W (swa_new
// optional), and, where (t+1) mod m == 0, the indexer key of entry
// (t+1)/m - 1: copied from kI_new, or computed by the key compressor from
// its staging ring (`keys`, ring mode).  Sequences with t < 0 are skipped,
// and so is an entry past n_cap.
struct DecodeAppend {
  const int32_t* q_pos;
  int B, W, m;
  const uint16_t* swa_new;  // [B][kDim] bf16, or null
  uint16_t* swa_ring;       // [B][W][kDim] bf16
  const uint8_t* kI_new;    // [B][kIdxDim] e4m3, or null
  uint8_t* kI;              // [B][n_cap][kIdxDim] e4m3
  int64_t n_cap;
};
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t stream, const DecodeAppend* append = nullptr,
                        const CompressArgs* keys = nullptr);

// ---- top-k -------------------------------------------------------------------------
struct TopkArgs {
  const float* scores;      // fp32, or bf16 (uint16) with bf16_scores
  int64_t score_ld;
  int bf16_scores;
  const uint32_t* hist;     // [B*Q][2048] key first-digit counts from the indexer
  const int32_t* q_pos;
  int64_t pos_base;
  int B, Q, m, k;
  int64_t n_cap;
  int32_t* idx_out;         // [B][Q][k]
  float* score_out;         // [B][Q][k] or null
  uint32_t* bits;           // [B*Q][bits_ld] selected-position bitmap of rows longer than the
                            // on-chip bitmaps hold (scratch, never read before it is written)
  int64_t bits_ld;          // topk_bits_ld(n_cap)
  // Row extent: the visible entries V(t) by default; with vis_shift = s the
  // ceil(V/2^s) blocks of 2^s entries (block scores); with a pool the row's
  // valid pool slots, and the output positions map to entries through it.
  int vis_shift;
  const int32_t* pool;      // [B*Q][pool_ld] or null
  int pool_blocks;
  int64_t pool_ld;
  unsigned* status;
};
// Words per row of the top-k position bitmaps (a multiple of 4).
int64_t topk_bits_ld(int64_t n_cap);
// ride_along: optional decode-mode (mode 1) compressor arguments for the same
// B sequences, computed by extra CTAs of the same launch (m for which
// topk_can_carry_compress holds).
bool topk_can_carry_compress(int m);
// second: an optional independent selection run by the same launch (its
// sequences after a's along the grid); not together with a ride-along.
cudaError_t launch_topk(const TopkArgs& a, const CompressArgs* ride_along, cudaStream_t stream,
                        const TopkArgs* second = nullptr);

// ---- sparse attention (tcgen05, bf16) ------------------------------------------------
struct AttnArgs {
  const int32_t* q_pos;     // [B][Q] or null (then pos_base + q)
  int64_t pos_base;
  const uint16_t* q;        // [B][Q][64][512]
  const uint16_t* kv;       // [B][n_cap][512] bf16 (unused with kv_fp4)
  const uint8_t* kv_fp4;    // [B][n_cap][kFp4Entry] FP4 entries, or null
  int64_t n_cap;
  const int32_t* idx;       // [B][Q][k] (sparse)
  int k;
  int dense;                // 1: the rows are every visible entry 0 .. V(t)-1 (idx unused)
  int m;                    // dense: V(t) = floor((t+1)/m), at most n_cap
  const uint16_t* swa;
  int swa_mode;             // 0 ring [B][W][512]; 1 linear [B][swa_len][512]
  int64_t swa_len;
  const int32_t* swa_pos0;  // [B] (mode 1) or null (then swa_pos0_base)
  int64_t swa_pos0_base;
  int W;
  const float* sink;        // [64]
  uint16_t* out;            // [B][Q][64][512]
  float* lse;               // [B][Q][64] or null
  int B, Q;
  float sm_scale;
  // Workspace of the split-KV path: per query gsplit_cap slices of raw
  // O [64][512] fp32, then per query gsplit_cap (max, sum) [2][64] fp32;
  // null: no such path.
  float* part_o;
  float* part_ml;
  int gsplit_cap;
  int inverse_rope;            // 1: rotate the output's RoPE channels back by -t
  uint64_t rope_turns[kRope / 2];  // theta^(-2j/R) / (2 pi) * 2^64 (fill_rope_turns)
  // 1: the call's first kernel was a launch_zero kernel (which lets its
  // dependents start only once its own predecessor has completed) and no
  // kernel since writes q, q_pos or sink: the kernel loads them before
  // waiting for its predecessor
  int early;
  unsigned* status;
  // set by launch_sparse_attn: tensor maps of the window buffer and of the
  // bf16 cache exist, so tiles of 128 consecutive present rows load by TMA
  int tma_swa, tma_kv;
};
constexpr int kMaxGSplit = 16;  // split-KV slices per query at most
constexpr size_t kGSplitSliceBytes = static_cast<size_t>(kHeads * kDim + 2 * kHeads) * 4;  // raw O + (max, sum)
// Slices per query of the split-KV path for `queries` queries on a GPU of
// `sms` SMs: one wave of one CTA per slice, at most kMaxGSplit; 0 when fewer
// than 2 fit (the cluster path then serves the launch).
inline int attn_split_slices(int64_t queries, int sms) {
  if (queries <= 0 || sms <= 0) return 0;
  const int64_t g = sms / queries < kMaxGSplit ? sms / queries : kMaxGSplit;
  return g >= 2 ? static_cast<int>(g) : 0;
}
inline size_t attn_split_bytes(int64_t queries, int sms) {
  return static_cast<size_t>(queries) * attn_split_slices(queries, sms) * kGSplitSliceBytes;
}
cudaError_t launch_sparse_attn(const AttnArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode, cudaStream_t stream);

// ---- FP4 cache entries -------------------------------------------------------------
// bf16 rows of kDim (row r at in + r*in_stride) -> FP4 entries of kFp4Entry
// bytes (entry r at out + r*out_stride).
// bf16 rows of 128 (row j of sequence b at in + b*in_stride_b + j*128) ->
// FP4 indexer rows: codes at codes + b*codes_stride_b + e*64 and E8M0 scales
// in 512-byte atoms at sf + b*sf_stride_b (e = entry0 + j, layout of
// IndexArgs::kI_sf); zero_pad: also zero bytes 8..15 of each atom line (the
// query records, whose 64 rows fill half an atom).
struct IndexFp4Rows {
  const uint16_t* in;
  int64_t in_stride_b;
  int B, n_rows;
  int64_t entry0;
  uint8_t* codes;
  int64_t codes_stride_b;
  uint8_t* sf;
  int64_t sf_stride_b;
  int zero_pad;
};
cudaError_t launch_quantize_index_fp4(const IndexFp4Rows& a, cudaStream_t stream);
cudaError_t launch_quantize_kv_fp4(int64_t n_rows, const uint16_t* in, int64_t in_stride, uint8_t* out,
                                   int64_t out_stride, cudaStream_t stream);

}  // namespace csa
