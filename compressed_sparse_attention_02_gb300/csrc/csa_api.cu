// C ABI of libcsa (declared in include/csa.h): host-side argument checks,
// workspace sizing, and the launch sequences of the single-stage and layer
// calls.  No call allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/csa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {
std::atomic<uint64_t> g_launches{0};
}
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace csa

namespace {

// Device status word: kernels OR error bits into it, csa_check_status reads
// and clears it.  One per device (module globals are per context).  The
// words after it hold the test faults and test wait limit (see ptx.cuh),
// zero unless csa_test_set_wait_fault set them.
__device__ unsigned g_status_word[4];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_status_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

unsigned* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// Stage tracing (csa_set_trace_events): events recorded between the stages
// of the layer calls.
cudaEvent_t g_trace[5] = {};
bool g_trace_on = false;

void trace(int stage, cudaStream_t st) {
  if (g_trace_on) cudaEventRecord(g_trace[stage], st);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
bool ok_opt(const void* p) { return p == nullptr || aligned16(p); }

// The overlapped compressor (and the layer calls that run it) exist for the
// CSA block sizes 1..8.
csa_status check_overlapped(const csa_params* p) { return p->m <= 8 ? CSA_OK : CSA_ERR_UNSUPPORTED; }

// Calls that write or read the cache as bf16 rows.
csa_status check_bf16_cache(const csa_params* p) { return p->kv_format == 0 ? CSA_OK : CSA_ERR_UNSUPPORTED; }

// Dimensions the kernels are built for; anything else is unsupported.
csa_status check_params(const csa_params* p) {
  if (!p) return CSA_ERR_INVALID_ARG;
  if (p->n_heads != csa::kHeads || p->head_dim != csa::kDim || p->rope_dim != csa::kRope ||
      p->idx_heads != csa::kIdxHeads || p->idx_dim != csa::kIdxDim)
    return CSA_ERR_UNSUPPORTED;
  // block sizes: the overlapped CSA compressor 1..8 (checked by its calls),
  // the single-stream HCA / CSA2 compressor up to 128
  if (p->m < 1 || p->m > csa::kMaxSingleM || (p->m & (p->m - 1)) != 0) return CSA_ERR_UNSUPPORTED;
  if (p->topk < 1 || p->topk > csa::kMaxTopk) return CSA_ERR_UNSUPPORTED;
  if (p->swa_window < 1 || p->swa_window > csa::kMaxWindow) return CSA_ERR_UNSUPPORTED;
  if (!(p->rope_theta > 0.f) || !(p->rms_eps >= 0.f) || !isfinite(p->sm_scale)) return CSA_ERR_INVALID_ARG;
  if (p->inverse_rope != 0 && p->inverse_rope != 1) return CSA_ERR_INVALID_ARG;
  if (p->kv_format != 0 && p->kv_format != 1) return CSA_ERR_UNSUPPORTED;
  if (p->bf16_scores != 0 && p->bf16_scores != 1) return CSA_ERR_INVALID_ARG;
  if (p->index_format != 0 && p->index_format != 1) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

struct IndexWs {
  size_t scores_off, hist_off, bits_off, total;
  size_t zero_bytes;  // the digit counts, cleared before each call
  int64_t score_ld, bits_ld;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Scratch of the indexer and top-k: scores [rows][score_ld] fp32; per row the
// counts of the 2048 score-key first digits (cleared by one launch before
// the indexer adds to them); the position bitmaps of rows too long for the
// top-k's on-chip bitmaps.
bool index_workspace(int64_t rows, int64_t n_cap, IndexWs* w) {
  if (rows < 0 || n_cap < 0 || static_cast<double>(rows) * static_cast<double>(n_cap) > 1e13) return false;
  w->score_ld = static_cast<int64_t>(round_up(static_cast<size_t>(n_cap), 8));  // 16-byte rows as bf16 too
  w->bits_ld = csa::topk_bits_ld(n_cap);
  const size_t R = static_cast<size_t>(rows);
  w->scores_off = 0;
  size_t off = round_up(R * w->score_ld * 4, 256);
  w->hist_off = off;
  w->zero_bytes = R * 2048 * 4;
  off = round_up(off + w->zero_bytes, 256);
  w->bits_off = off;
  off = round_up(off + R * w->bits_ld * 4, 256);
  w->total = off;
  return true;
}

csa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

// The hierarchical indexer's side of a call: a pool to score (Reindex layer)
// or a pool to produce (Full layer), of `blocks` blocks.
struct PoolSpec {
  const int32_t* in = nullptr;
  int32_t* out = nullptr;
  int blocks = 0;
};

// Full layer scratch: the entries' indexer scratch, then the same layout for
// the ceil(n_cap/8) block scores.
bool pool_workspace(int64_t rows, int64_t n_cap, IndexWs* w, IndexWs* wb, size_t* total) {
  if (!index_workspace(rows, n_cap, w) || !index_workspace(rows, (n_cap + 7) / 8, wb))
    return false;
  *total = w->total + wb->total;
  return true;
}

bool pool_blocks_ok(int32_t blocks) {
  return blocks >= csa::kPoolTileBlocks && blocks <= csa::kMaxTopk && blocks % csa::kPoolTileBlocks == 0;
}

// Fills the top-k arguments that point into one IndexWs.
void topk_scratch(csa::TopkArgs* ta, uint8_t* base, const IndexWs& w) {
  ta->scores = reinterpret_cast<const float*>(base + w.scores_off);
  ta->score_ld = w.score_ld;
  ta->hist = reinterpret_cast<const uint32_t*>(base + w.hist_off);
  ta->bits = reinterpret_cast<uint32_t*>(base + w.bits_off);
  ta->bits_ld = w.bits_ld;
}

// Shared body of csa_index_topk, the hierarchical indexer calls and the
// layer calls.
csa_status run_index_topk(const csa_params* p, int32_t B, int32_t Q, const int32_t* q_pos, int64_t pos_base,
                          const uint8_t* qI, const uint16_t* wI, const uint8_t* kI, int64_t n_cap,
                          int32_t* idx_out, float* score_out, void* ws, size_t ws_bytes, cudaStream_t st,
                          bool traced = false, bool zeroed = false,
                          const csa::CompressArgs* ride_along = nullptr, const PoolSpec* pool = nullptr,
                          bool standalone = false, bool after_zero = false) {
  const int64_t rows = static_cast<int64_t>(B) * Q;
  IndexWs w, wb;
  size_t need = 0;
  bool sized;
  if (pool && pool->in) {
    sized = index_workspace(rows, static_cast<int64_t>(pool->blocks) * csa::kPoolBlock, &w);
    need = w.total;
  } else if (pool && pool->out) {
    sized = pool_workspace(rows, n_cap, &w, &wb, &need);
  } else {
    sized = index_workspace(rows, n_cap, &w);
    need = w.total;
  }
  if (!sized) return CSA_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < need || !aligned16(ws)) return CSA_ERR_WORKSPACE;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  unsigned* status = status_ptr();
  if (!enc || !status) return CSA_ERR_CUDA;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  uint8_t* wsb_blk = wsb + w.total;  // Full layer: the block scores' scratch
  float* scores = reinterpret_cast<float*>(wsb + w.scores_off);
  uint32_t* hist = reinterpret_cast<uint32_t*>(wsb + w.hist_off);
  if (!zeroed && csa::launch_zero(hist, w.zero_bytes, st) != cudaSuccess) return CSA_ERR_CUDA;
  if (pool && pool->out && csa::launch_zero(wsb_blk + wb.hist_off, wb.zero_bytes, st) != cudaSuccess)
    return CSA_ERR_CUDA;
  // a call of its own (not inside a layer call) traces from its indexer on
  const bool own = traced && (pool || standalone);
  if (own) trace(1, st);

  csa::IndexArgs ia = {};
  ia.qI = qI;
  ia.wI = wI;
  ia.kI = kI;
  ia.q_pos = q_pos;
  ia.pos_base = pos_base;
  ia.B = B;
  ia.Q = Q;
  ia.m = p->m;
  ia.n_cap = n_cap;
  ia.scores = scores;
  ia.score_ld = w.score_ld;
  ia.bf16_scores = p->bf16_scores;
  ia.hist = hist;
  if (p->index_format == 1) {  // FP4: the scale planes follow the code planes
    ia.fp4 = 1;
    ia.kI_sf = kI + static_cast<int64_t>(B) * n_cap * (csa::kIdxDim / 2);
    ia.kI_sf_ld = (n_cap + 127) / 128 * 512;
    ia.qI_sf = qI + rows * csa::kIdxHeads * (csa::kIdxDim / 2);
  }
  if (pool && pool->in) {
    ia.pool = pool->in;
    ia.pool_blocks = pool->blocks;
    ia.pool_ld = pool->blocks;
  }
  if (pool && pool->out) {
    ia.block_scores = reinterpret_cast<float*>(wsb_blk + wb.scores_off);
    ia.block_ld = wb.score_ld;
    ia.block_hist = reinterpret_cast<uint32_t*>(wsb_blk + wb.hist_off);
  }
  // the indexer may start on its key tiles before the zeroing kernel right
  // before it has finished (not across a trace event, not in pool mode)
  ia.early = (!zeroed || after_zero) && !own && !(pool && pool->in);
  ia.status = status;
  csa_status s = cuda_status(csa::launch_index_scores(ia, enc, st));
  if (s != CSA_OK) return s;
  if (traced) trace(2, st);

  csa::TopkArgs ta = {};
  topk_scratch(&ta, wsb, w);
  ta.bf16_scores = p->bf16_scores;
  ta.q_pos = q_pos;
  ta.pos_base = pos_base;
  ta.B = B;
  ta.Q = Q;
  ta.m = p->m;
  ta.k = p->topk;
  ta.n_cap = n_cap;
  ta.idx_out = idx_out;
  ta.score_out = score_out;
  if (pool && pool->in) {
    ta.pool = pool->in;
    ta.pool_blocks = pool->blocks;
    ta.pool_ld = pool->blocks;
  }
  ta.status = status;
  csa::TopkArgs tb = {};
  if (pool && pool->out) {  // the pool, in the same launch: the top `blocks` block scores, ids ascending
    tb = ta;
    topk_scratch(&tb, wsb_blk, wb);
    tb.k = pool->blocks;
    tb.vis_shift = 3;
    tb.bf16_scores = 0;  // the block scores stay fp32
    tb.idx_out = pool->out;
    tb.score_out = nullptr;
  }
  s = cuda_status(csa::launch_topk(ta, ride_along, st, pool && pool->out ? &tb : nullptr));
  if (s == CSA_OK && own) trace(3, st);
  return s;
}

csa_status run_attn(const csa_params* p, int32_t B, int32_t Q, const int32_t* q_pos, int64_t pos_base,
                    const uint16_t* q, const void* kv, int64_t n_cap, const int32_t* idx, const uint16_t* swa,
                    int32_t swa_mode, int64_t swa_len, const int32_t* swa_pos0, int64_t swa_pos0_base,
                    const float* sink, uint16_t* out, float* lse, cudaStream_t st, bool dense = false,
                    void* split_ws = nullptr, size_t split_ws_bytes = 0, bool early = false) {
  unsigned* status = status_ptr();
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!status || !enc) return CSA_ERR_CUDA;
  csa::AttnArgs aa = {};
  aa.q_pos = q_pos;
  aa.pos_base = pos_base;
  aa.q = q;
  if (p->kv_format == 1)
    aa.kv_fp4 = static_cast<const uint8_t*>(kv);
  else
    aa.kv = static_cast<const uint16_t*>(kv);
  aa.n_cap = n_cap;
  aa.idx = idx;
  aa.k = p->topk;
  aa.dense = dense ? 1 : 0;
  aa.m = p->m;
  // the split-KV path, with as many slices per query as the workspace holds
  const int64_t queries = static_cast<int64_t>(B) * Q;
  if (split_ws && aligned16(split_ws) && queries > 0) {
    int64_t cap = static_cast<int64_t>(split_ws_bytes / (static_cast<size_t>(queries) * csa::kGSplitSliceBytes));
    cap = cap < csa::kMaxGSplit ? cap : csa::kMaxGSplit;
    if (cap >= 2) {
      aa.part_o = static_cast<float*>(split_ws);
      aa.part_ml = aa.part_o + queries * cap * csa::kHeads * csa::kDim;
      aa.gsplit_cap = static_cast<int>(cap);
    }
  }
  aa.swa = swa;
  aa.swa_mode = swa_mode;
  aa.swa_len = swa_len;
  aa.swa_pos0 = swa_pos0;
  aa.swa_pos0_base = swa_pos0_base;
  aa.W = p->swa_window;
  aa.sink = sink;
  aa.out = out;
  aa.lse = lse;
  aa.B = B;
  aa.Q = Q;
  aa.sm_scale = p->sm_scale;
  aa.inverse_rope = p->inverse_rope;
  csa::fill_rope_turns(static_cast<double>(p->rope_theta), aa.rope_turns);
  aa.early = early ? 1 : 0;
  aa.status = status;
  return cuda_status(csa::launch_sparse_attn(aa, enc, st));
}

csa::CompressArgs compress_args(const csa_params* p, int mode, int32_t B, int64_t n_new, int64_t entry0,
                                const uint16_t* Ca, const uint16_t* Za, const uint16_t* Cb, const uint16_t* Zb,
                                const uint16_t* Cb_prev, const uint16_t* Zb_prev, const uint16_t* Ba,
                                const uint16_t* Bb, const uint16_t* rms_w, uint16_t* kv_out, int64_t kv_stride_b,
                                int64_t n_cap, const int32_t* q_pos, unsigned* status) {
  csa::CompressArgs ca = {};
  ca.mode = mode;
  ca.B = B;
  ca.m = p->m;
  ca.n_new = n_new;
  ca.entry0 = entry0;
  ca.Ca = Ca;
  ca.Za = Za;
  ca.Cb = Cb;
  ca.Zb = Zb;
  ca.Cb_prev = Cb_prev;
  ca.Zb_prev = Zb_prev;
  ca.Ba = Ba;
  ca.Bb = Bb;
  ca.rms_w = rms_w;
  ca.kv_out = kv_out;
  ca.kv_stride_b = kv_stride_b;
  ca.n_cap = n_cap;
  ca.q_pos = q_pos;
  ca.rope_theta = static_cast<double>(p->rope_theta);
  ca.rms_eps = p->rms_eps;
  ca.status = status;
  return ca;
}

csa_status run_compress(const csa_params* p, int mode, int32_t B, int64_t n_new, int64_t entry0,
                        const uint16_t* Ca, const uint16_t* Za, const uint16_t* Cb, const uint16_t* Zb,
                        const uint16_t* Cb_prev, const uint16_t* Zb_prev, const uint16_t* Ba,
                        const uint16_t* Bb, const uint16_t* rms_w, uint16_t* kv_out, int64_t kv_stride_b,
                        int64_t n_cap, const int32_t* q_pos, cudaStream_t st, uint8_t* fp4_out = nullptr,
                        int64_t fp4_stride_b = 0, const csa::CompressArgs* keys = nullptr) {
  unsigned* status = status_ptr();
  if (!status) return CSA_ERR_CUDA;
  csa::CompressArgs ca = compress_args(p, mode, B, n_new, entry0, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, rms_w,
                                       kv_out, kv_stride_b, n_cap, q_pos, status);
  ca.kv_fp4_out = fp4_out;
  ca.fp4_stride_b = fp4_stride_b;
  return cuda_status(csa::launch_compress(ca, st, keys));
}

// The key compressor's arguments for the layer calls: mode 1 (decode ring)
// or 0 (a chunk's rows), E4M3 keys into kI [B][n_cap][128].
csa::CompressArgs key_args(const csa_params* p, int mode, int32_t B, int64_t n_new, int64_t entry0,
                           const csa_index_key_src& k, uint8_t* kI, int64_t n_cap, const int32_t* q_pos,
                           unsigned* status) {
  csa::CompressArgs ka = compress_args(p, mode, B, n_new, entry0, k.CIa, k.ZIa, k.CIb, k.ZIb,
                                       mode == 0 ? k.CIb_prev : nullptr, mode == 0 ? k.ZIb_prev : nullptr, k.BIa,
                                       k.BIb, k.rms_wI, nullptr, n_cap * csa::kIdxDim, n_cap, q_pos, status);
  ka.key_out = kI;
  return ka;
}

bool key_src_ok(const csa_index_key_src* k, bool prefill, int64_t pos0) {
  if (!k || !ok_ptr(k->CIa) || !ok_ptr(k->ZIa) || !ok_ptr(k->CIb) || !ok_ptr(k->ZIb) || !ok_ptr(k->BIa) ||
      !ok_ptr(k->BIb) || !ok_ptr(k->rms_wI))
    return false;
  if (!prefill) return true;
  return (pos0 > 0) == (k->CIb_prev != nullptr) && (k->CIb_prev == nullptr) == (k->ZIb_prev == nullptr) &&
         ok_opt(k->CIb_prev) && ok_opt(k->ZIb_prev);
}

bool n_cap_ok(int64_t n_cap) { return n_cap >= 1 && n_cap <= (int64_t(1) << 30); }

// Scratch of csa_index_topk_static: a fixed device array, so that callers
// who cannot allocate device memory can still run the indexer.  Host code
// sees only a stand-in for this symbol; its device address is looked up once
// per device (with that device current) and passed to the kernels.
__device__ __align__(256) unsigned char g_static_scratch[CSA_STATIC_SCRATCH_BYTES];
void* g_static_scratch_ptr[kMaxDevices] = {};

void* static_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_static_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_static_scratch_ptr[dev] = p;
  }
  return g_static_scratch_ptr[dev];
}

}  // namespace

extern "C" {

void csa_default_params(csa_params* p) {
  if (!p) return;
  p->m = 4;
  p->n_heads = 64;
  p->head_dim = 512;
  p->rope_dim = 64;
  p->idx_heads = 64;
  p->idx_dim = 128;
  p->topk = 512;
  p->swa_window = 128;
  p->rope_theta = 10000.f;
  p->rms_eps = 1e-6f;
  p->sm_scale = 0.044194173824159216f;  // 1/sqrt(512)
  p->inverse_rope = 0;
  p->kv_format = 0;
  p->bf16_scores = 0;
  p->index_format = 0;
}

// SMs of the current device (0 without one): the split-KV scratch is sized
// for one wave of its slices.
int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return sms;
}

size_t csa_workspace_size(int32_t op, const csa_params* p, int32_t B, int32_t Q, int64_t n_cap) {
  if (check_params(p) != CSA_OK || B < 0 || Q < 0 || !n_cap_ok(n_cap)) return 0;
  IndexWs w;
  const int sms = device_sms();
  switch (op) {
    case CSA_OP_COMPRESS:
      return 16;  // no scratch needed; a non-zero size keeps callers uniform
    case CSA_OP_SPARSE_ATTN: {  // the split-KV partials
      const size_t a = csa::attn_split_bytes(static_cast<int64_t>(B) * Q, sms);
      return a > 16 ? a : 16;
    }
    case CSA_OP_INDEX_TOPK:
      return index_workspace(static_cast<int64_t>(B) * Q, n_cap, &w) ? w.total : 0;
    case CSA_OP_LAYER_PREFILL:  // the indexer's scratch, then the attention's
      return index_workspace(static_cast<int64_t>(B) * Q, n_cap, &w)
                 ? round_up(w.total, 256) + csa::attn_split_bytes(static_cast<int64_t>(B) * Q, sms)
                 : 0;
    case CSA_OP_LAYER_DECODE:
      return index_workspace(static_cast<int64_t>(B), n_cap, &w)
                 ? round_up(w.total, 256) + csa::attn_split_bytes(B, sms)
                 : 0;
    case CSA_OP_HCA_LAYER_DECODE: {  // the attention's split-KV partials
      const size_t a = csa::attn_split_bytes(B, sms);
      return a > 16 ? a : 16;
    }
    case CSA_OP_INDEX_TOPK_POOL: {
      IndexWs wb;
      size_t total = 0;
      return pool_workspace(static_cast<int64_t>(B) * Q, n_cap, &w, &wb, &total) ? total : 0;
    }
    case CSA_OP_REINDEX_TOPK:  // sized for the largest pool
      return index_workspace(static_cast<int64_t>(B) * Q, static_cast<int64_t>(csa::kMaxTopk) * csa::kPoolBlock, &w)
                 ? w.total
                 : 0;
    default:
      return 0;
  }
}

csa_status csa_compress(const csa_params* p, int32_t B, int32_t n_new, int64_t entry0, const uint16_t* Ca,
                        const uint16_t* Za, const uint16_t* Cb, const uint16_t* Zb, const uint16_t* Cb_prev,
                        const uint16_t* Zb_prev, const uint16_t* Ba, const uint16_t* Bb, const uint16_t* rms_w,
                        uint16_t* kv_out, int64_t kv_stride_b, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if ((s = check_bf16_cache(p)) != CSA_OK) return s;
  if ((s = check_overlapped(p)) != CSA_OK) return s;
  if (B < 0 || n_new < 0 || entry0 < 0 || B > 65535) return CSA_ERR_INVALID_ARG;
  if (B == 0 || n_new == 0) return CSA_OK;
  if (!ok_ptr(Ca) || !ok_ptr(Za) || !ok_ptr(Cb) || !ok_ptr(Zb) || !ok_ptr(Ba) || !ok_ptr(Bb) ||
      !ok_ptr(rms_w) || !ok_ptr(kv_out))
    return CSA_ERR_INVALID_ARG;
  if ((entry0 > 0) != (Cb_prev != nullptr) || (Cb_prev == nullptr) != (Zb_prev == nullptr) || !ok_opt(Cb_prev) ||
      !ok_opt(Zb_prev))
    return CSA_ERR_INVALID_ARG;
  if (kv_stride_b < (entry0 + n_new) * csa::kDim && B > 1) return CSA_ERR_INVALID_ARG;
  if (kv_stride_b % 8 != 0) return CSA_ERR_INVALID_ARG;
  return run_compress(p, 0, B, n_new, entry0, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, rms_w, kv_out,
                      kv_stride_b, entry0 + n_new, nullptr, static_cast<cudaStream_t>(stream));
}

csa_status csa_compress_indexer_keys(const csa_params* p, int32_t B, int32_t n_new, int64_t entry0,
                                     const uint16_t* CIa, const uint16_t* ZIa, const uint16_t* CIb,
                                     const uint16_t* ZIb, const uint16_t* CIb_prev, const uint16_t* ZIb_prev,
                                     const uint16_t* BIa, const uint16_t* BIb, const uint16_t* rms_wI,
                                     uint8_t* kI_out, int64_t kI_stride_b, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if ((s = check_overlapped(p)) != CSA_OK) return s;
  if (p->index_format != 0) return CSA_ERR_UNSUPPORTED;  // this compressor writes E4M3 keys
  if (B < 0 || n_new < 0 || entry0 < 0 || B > 65535) return CSA_ERR_INVALID_ARG;
  if (B == 0 || n_new == 0) return CSA_OK;
  if (!ok_ptr(CIa) || !ok_ptr(ZIa) || !ok_ptr(CIb) || !ok_ptr(ZIb) || !ok_ptr(BIa) || !ok_ptr(BIb) ||
      !ok_ptr(rms_wI) || !ok_ptr(kI_out))
    return CSA_ERR_INVALID_ARG;
  if ((entry0 > 0) != (CIb_prev != nullptr) || (CIb_prev == nullptr) != (ZIb_prev == nullptr) ||
      !ok_opt(CIb_prev) || !ok_opt(ZIb_prev))
    return CSA_ERR_INVALID_ARG;
  if (kI_stride_b < (entry0 + n_new) * csa::kIdxDim && B > 1) return CSA_ERR_INVALID_ARG;
  if (kI_stride_b % 16 != 0) return CSA_ERR_INVALID_ARG;
  unsigned* status = status_ptr();
  if (!status) return CSA_ERR_CUDA;
  csa::CompressArgs ca = compress_args(p, 0, B, n_new, entry0, CIa, ZIa, CIb, ZIb, CIb_prev, ZIb_prev, BIa, BIb,
                                       rms_wI, nullptr, kI_stride_b, entry0 + n_new, nullptr, status);
  ca.key_out = kI_out;
  return cuda_status(csa::launch_index_keys(ca, static_cast<cudaStream_t>(stream)));
}

csa_status csa_compress_single(const csa_params* p, int32_t B, int32_t n_new, int64_t entry0, const uint16_t* C,
                               const uint16_t* Z, const uint16_t* bias, const uint16_t* rms_w, uint16_t* kv_out,
                               int64_t kv_stride_b, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if ((s = check_bf16_cache(p)) != CSA_OK) return s;
  if (B < 0 || n_new < 0 || entry0 < 0 || B > 65535) return CSA_ERR_INVALID_ARG;
  if (B == 0 || n_new == 0) return CSA_OK;
  if (!ok_ptr(C) || !ok_ptr(Z) || !ok_opt(bias) || !ok_ptr(rms_w) || !ok_ptr(kv_out)) return CSA_ERR_INVALID_ARG;
  if (kv_stride_b < (entry0 + n_new) * csa::kDim && B > 1) return CSA_ERR_INVALID_ARG;
  if (kv_stride_b % 8 != 0) return CSA_ERR_INVALID_ARG;
  unsigned* status = status_ptr();
  if (!status) return CSA_ERR_CUDA;
  csa::CompressArgs ca = compress_args(p, 0, B, n_new, entry0, C, Z, nullptr, nullptr, nullptr, nullptr, bias, nullptr,
                                       rms_w, kv_out, kv_stride_b, entry0 + n_new, nullptr, status);
  return cuda_status(csa::launch_compress_single(ca, static_cast<cudaStream_t>(stream)));
}

csa_status csa_compress_single_step(const csa_params* p, int32_t B, const int32_t* q_pos, const uint16_t* C,
                                    const uint16_t* Z, const uint16_t* bias, const uint16_t* rms_w, float* state,
                                    uint16_t* kv_out, int64_t kv_stride_b, int64_t n_cap, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if ((s = check_bf16_cache(p)) != CSA_OK) return s;
  if (B < 0 || B > 65535 || !n_cap_ok(n_cap)) return CSA_ERR_INVALID_ARG;
  if (B == 0) return CSA_OK;
  if (!ok_ptr(q_pos) || !ok_ptr(C) || !ok_ptr(Z) || !ok_opt(bias) || !ok_ptr(rms_w) || !ok_ptr(state) ||
      !ok_ptr(kv_out))
    return CSA_ERR_INVALID_ARG;
  if (kv_stride_b < n_cap * csa::kDim && B > 1) return CSA_ERR_INVALID_ARG;
  if (kv_stride_b % 8 != 0) return CSA_ERR_INVALID_ARG;
  unsigned* status = status_ptr();
  if (!status) return CSA_ERR_CUDA;
  csa::CompressArgs ca = compress_args(p, 1, B, 0, 0, C, Z, nullptr, nullptr, nullptr, nullptr, bias, nullptr, rms_w,
                                       kv_out, kv_stride_b, n_cap, q_pos, status);
  ca.state = state;
  return cuda_status(csa::launch_compress_single(ca, static_cast<cudaStream_t>(stream)));
}

csa_status csa_quantize_kv_fp4(int64_t n_rows, const uint16_t* in, int64_t in_stride, uint8_t* out,
                               int64_t out_stride, void* stream) {
  if (n_rows < 0 || n_rows > (int64_t(1) << 40)) return CSA_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA_OK;
  if (!ok_ptr(in) || !ok_ptr(out)) return CSA_ERR_INVALID_ARG;
  if (in_stride < csa::kDim || in_stride % 8 != 0 || out_stride < csa::kFp4Entry || out_stride % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  return cuda_status(csa::launch_quantize_kv_fp4(n_rows, in, in_stride, out, out_stride,
                                                 static_cast<cudaStream_t>(stream)));
}

csa_status csa_quantize_index_keys_fp4(int32_t B, int32_t n_new, int64_t entry0, const uint16_t* in,
                                       int64_t in_stride_b, uint8_t* kI, int64_t n_cap, void* stream) {
  if (B < 0 || n_new < 0 || entry0 < 0 || B > 65535 || !n_cap_ok(n_cap) || entry0 + n_new > n_cap)
    return CSA_ERR_INVALID_ARG;
  if (B == 0 || n_new == 0) return CSA_OK;
  if (!ok_ptr(in) || !ok_ptr(kI) || in_stride_b % 8 != 0 ||
      (B > 1 && in_stride_b < static_cast<int64_t>(n_new) * csa::kIdxDim))
    return CSA_ERR_INVALID_ARG;
  csa::IndexFp4Rows a = {};
  a.in = in;
  a.in_stride_b = in_stride_b;
  a.B = B;
  a.n_rows = n_new;
  a.entry0 = entry0;
  a.codes = kI;
  a.codes_stride_b = n_cap * (csa::kIdxDim / 2);
  a.sf = kI + static_cast<int64_t>(B) * n_cap * (csa::kIdxDim / 2);
  a.sf_stride_b = (n_cap + 127) / 128 * 512;
  return cuda_status(csa::launch_quantize_index_fp4(a, static_cast<cudaStream_t>(stream)));
}

csa_status csa_quantize_index_query_fp4(int64_t n_q, const uint16_t* in, uint8_t* qI, void* stream) {
  if (n_q < 0 || n_q > (int64_t(1) << 31) - 1) return CSA_ERR_INVALID_ARG;
  if (n_q == 0) return CSA_OK;
  if (!ok_ptr(in) || !ok_ptr(qI)) return CSA_ERR_INVALID_ARG;
  csa::IndexFp4Rows a = {};  // a query is a "sequence" of 64 head rows sharing one atom
  a.in = in;
  a.in_stride_b = static_cast<int64_t>(csa::kIdxHeads) * csa::kIdxDim;
  a.B = static_cast<int>(n_q);
  a.n_rows = csa::kIdxHeads;
  a.codes = qI;
  a.codes_stride_b = csa::kIdxHeads * (csa::kIdxDim / 2);
  a.sf = qI + n_q * csa::kIdxHeads * (csa::kIdxDim / 2);
  a.sf_stride_b = 512;
  a.zero_pad = 1;
  return cuda_status(csa::launch_quantize_index_fp4(a, static_cast<cudaStream_t>(stream)));
}

csa_status csa_index_topk(const csa_params* p, int32_t B, int32_t Q, const int32_t* q_pos, const uint8_t* qI,
                          const uint16_t* wI, const uint8_t* kI, int64_t n_cap, int32_t* idx_out, float* score_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if (B < 0 || Q < 0 || B > 65535 || Q > 65535 || !n_cap_ok(n_cap)) return CSA_ERR_INVALID_ARG;
  if (B == 0 || Q == 0) return CSA_OK;
  if (!ok_ptr(q_pos) || !ok_ptr(qI) || !ok_ptr(wI) || !ok_ptr(kI) || !ok_ptr(idx_out) || !ok_opt(score_out))
    return CSA_ERR_INVALID_ARG;
  return run_index_topk(p, B, Q, q_pos, 0, qI, wI, kI, n_cap, idx_out, score_out, workspace, workspace_bytes,
                        static_cast<cudaStream_t>(stream), g_trace_on, false, nullptr, nullptr, true);
}

csa_status csa_index_topk_static(const csa_params* p, int32_t B, int32_t Q, const int32_t* q_pos,
                                 const uint8_t* qI, const uint16_t* wI, const uint8_t* kI, int64_t n_cap,
                                 int32_t* idx_out, float* score_out, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if (B < 0 || Q < 0 || B > 65535 || Q > 65535 || !n_cap_ok(n_cap)) return CSA_ERR_INVALID_ARG;
  if (B == 0 || Q == 0) return CSA_OK;
  if (!ok_ptr(q_pos) || !ok_ptr(qI) || !ok_ptr(wI) || !ok_ptr(kI) || !ok_ptr(idx_out) || !ok_opt(score_out))
    return CSA_ERR_INVALID_ARG;
  IndexWs w;
  if (!index_workspace(static_cast<int64_t>(B) * Q, n_cap, &w)) return CSA_ERR_UNSUPPORTED;
  if (w.total > CSA_STATIC_SCRATCH_BYTES) return CSA_ERR_WORKSPACE;  // beyond the fixed array
  void* scratch = static_scratch();
  if (!scratch) return CSA_ERR_CUDA;
  return run_index_topk(p, B, Q, q_pos, 0, qI, wI, kI, n_cap, idx_out, score_out, scratch,
                        CSA_STATIC_SCRATCH_BYTES, static_cast<cudaStream_t>(stream), g_trace_on, false, nullptr,
                        nullptr, true);
}

csa_status csa_index_topk_pool(const csa_params* p, int32_t B, int32_t Q, const int32_t* q_pos, const uint8_t* qI,
                               const uint16_t* wI, const uint8_t* kI, int64_t n_cap, int32_t* idx_out,
                               float* score_out, int32_t pool_blocks, int32_t* pool_out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if (B < 0 || Q < 0 || B > 65535 || Q > 65535 || !n_cap_ok(n_cap)) return CSA_ERR_INVALID_ARG;
  if (!pool_blocks_ok(pool_blocks)) return CSA_ERR_UNSUPPORTED;
  if (B == 0 || Q == 0) return CSA_OK;
  if (!ok_ptr(q_pos) || !ok_ptr(qI) || !ok_ptr(wI) || !ok_ptr(kI) || !ok_ptr(idx_out) || !ok_opt(score_out) ||
      !ok_ptr(pool_out))
    return CSA_ERR_INVALID_ARG;
  PoolSpec ps;
  ps.out = pool_out;
  ps.blocks = pool_blocks;
  return run_index_topk(p, B, Q, q_pos, 0, qI, wI, kI, n_cap, idx_out, score_out, workspace, workspace_bytes,
                        static_cast<cudaStream_t>(stream), g_trace_on, false, nullptr, &ps);
}

csa_status csa_reindex_topk(const csa_params* p, int32_t B, int32_t Q, const int32_t* q_pos, const uint8_t* qI,
                            const uint16_t* wI, const uint8_t* kI, int64_t n_cap, const int32_t* pool,
                            int32_t pool_blocks, int32_t* idx_out, float* score_out, void* workspace,
                            size_t workspace_bytes, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if (B < 0 || Q < 0 || B > 65535 || Q > 65535 || !n_cap_ok(n_cap)) return CSA_ERR_INVALID_ARG;
  if (!pool_blocks_ok(pool_blocks)) return CSA_ERR_UNSUPPORTED;
  if (B == 0 || Q == 0) return CSA_OK;
  if (!ok_ptr(q_pos) || !ok_ptr(qI) || !ok_ptr(wI) || !ok_ptr(kI) || !ok_ptr(pool) || !ok_ptr(idx_out) ||
      !ok_opt(score_out))
    return CSA_ERR_INVALID_ARG;
  PoolSpec ps;
  ps.in = pool;
  ps.blocks = pool_blocks;
  return run_index_topk(p, B, Q, q_pos, 0, qI, wI, kI, n_cap, idx_out, score_out, workspace, workspace_bytes,
                        static_cast<cudaStream_t>(stream), g_trace_on, false, nullptr, &ps);
}

csa_status csa_sparse_attn(const csa_params* p, int32_t B, int32_t Q, const int32_t* q_pos, const uint16_t* q,
                           const void* kv_comp, int64_t n_cap, const int32_t* idx, const uint16_t* swa,
                           int32_t swa_mode, int64_t swa_len, const int32_t* swa_pos0, const float* sink,
                           uint16_t* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if (B < 0 || Q < 0 || B > 65535 || Q > 2147483647 || !n_cap_ok(n_cap)) return CSA_ERR_INVALID_ARG;
  if (B == 0 || Q == 0) return CSA_OK;
  if (!ok_ptr(q_pos) || !ok_ptr(q) || !ok_ptr(kv_comp) || !ok_opt(idx) || !ok_ptr(swa) || !ok_ptr(sink) ||
      !ok_ptr(out) || !ok_opt(lse))
    return CSA_ERR_INVALID_ARG;
  if (swa_mode == 0) {
    swa_len = p->swa_window;
  } else if (swa_mode == 1) {
    if (swa_len < 1 || !ok_ptr(swa_pos0)) return CSA_ERR_INVALID_ARG;
  } else {
    return CSA_ERR_INVALID_ARG;
  }
  return run_attn(p, B, Q, q_pos, 0, q, kv_comp, n_cap, idx, swa, swa_mode, swa_len, swa_pos0, 0, sink, out, lse,
                  static_cast<cudaStream_t>(stream), idx == nullptr, workspace, workspace_bytes);
}

namespace {
// One decode step; with `append`, the step's first kernel also writes the new
// window row and indexer key into the caches.
csa_status layer_decode(const csa_params* p, int32_t B, const int32_t* q_pos, const uint16_t* ring_Ca,
                        const uint16_t* ring_Za, const uint16_t* ring_Cb, const uint16_t* ring_Zb,
                        const uint16_t* Ba, const uint16_t* Bb, const uint16_t* rms_w, void* kv_comp,
                        int64_t n_cap, const uint8_t* kI, const uint8_t* qI, const uint16_t* wI,
                        const uint16_t* q, const uint16_t* swa_ring, const float* sink, int32_t* idx_out,
                        uint16_t* out, float* lse, void* workspace, size_t workspace_bytes, void* stream,
                        const csa::DecodeAppend* append, const csa_index_key_src* keys = nullptr,
                        uint8_t* kI_out = nullptr) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if ((s = check_overlapped(p)) != CSA_OK) return s;
  if (B < 0 || B > 65535 || !n_cap_ok(n_cap)) return CSA_ERR_INVALID_ARG;
  if (B == 0) return CSA_OK;
  if (!ok_ptr(q_pos) || !ok_ptr(ring_Ca) || !ok_ptr(ring_Za) || !ok_ptr(ring_Cb) || !ok_ptr(ring_Zb) ||
      !ok_ptr(Ba) || !ok_ptr(Bb) || !ok_ptr(rms_w) || !ok_ptr(kv_comp) || !ok_ptr(kI) || !ok_ptr(qI) ||
      !ok_ptr(wI) || !ok_ptr(q) || !ok_ptr(swa_ring) || !ok_ptr(sink) || !ok_ptr(idx_out) || !ok_ptr(out) ||
      !ok_opt(lse))
    return CSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  IndexWs w;
  if (!index_workspace(B, n_cap, &w)) return CSA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return CSA_ERR_WORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return CSA_ERR_CUDA;
  // the top-k counters are cleared first, so that the kernels follow one
  // another directly (programmatic launches); the same kernel stores the
  // step's new rows and computes its indexer key
  csa::CompressArgs ka = {};
  if (keys) ka = key_args(p, 1, B, 1, 0, *keys, kI_out, n_cap, q_pos, status);
  trace(0, st);
  if (csa::launch_zero(static_cast<uint8_t*>(workspace) + w.hist_off, w.zero_bytes, st, append,
                       keys ? &ka : nullptr) != cudaSuccess)
    return CSA_ERR_CUDA;
  // 1. emission of the entry that completes at this step (if any).  Only the
  //    attention reads it, so it is computed by extra CTAs of the top-k launch
  //    where that kernel can carry it, else by its own kernel first.
  // the cache holds bf16 rows or FP4 entries (p->kv_format); the compressor writes the same
  uint16_t* kv16 = p->kv_format ? nullptr : static_cast<uint16_t*>(kv_comp);
  csa::CompressArgs ca = compress_args(p, 1, B, 1, 0, ring_Ca, ring_Za, ring_Cb, ring_Zb, nullptr, nullptr, Ba, Bb,
                                       rms_w, kv16, n_cap * csa::kDim, n_cap, q_pos, status);
  if (p->kv_format) {
    ca.kv_fp4_out = static_cast<uint8_t*>(kv_comp);
    ca.fp4_stride_b = n_cap * csa::kFp4Entry;
  }
  const bool ride_along = csa::topk_can_carry_compress(p->m);
  if (!ride_along && (s = cuda_status(csa::launch_compress(ca, st))) != CSA_OK) return s;
  trace(1, st);
  // 2. indexer + top-k over the visible entries
  s = run_index_topk(p, B, 1, q_pos, 0, qI, wI, kI, n_cap, idx_out, nullptr, workspace, workspace_bytes, st, true,
                     true, ride_along ? &ca : nullptr, nullptr, false, ride_along);
  if (s != CSA_OK) return s;
  trace(3, st);
  // 3. sparse attention over the window ring and the selection
  const size_t attn_off = round_up(w.total, 256);
  s = run_attn(p, B, 1, q_pos, 0, q, kv_comp, n_cap, idx_out, swa_ring, 0, p->swa_window, nullptr, 0, sink, out,
               lse, st, false, static_cast<uint8_t*>(workspace) + attn_off,
               workspace_bytes > attn_off ? workspace_bytes - attn_off : 0, true);
  trace(4, st);
  return s;
}
}  // namespace

csa_status csa_layer_decode(const csa_params* p, int32_t B, const int32_t* q_pos, const uint16_t* ring_Ca,
                            const uint16_t* ring_Za, const uint16_t* ring_Cb, const uint16_t* ring_Zb,
                            const uint16_t* Ba, const uint16_t* Bb, const uint16_t* rms_w, void* kv_comp,
                            int64_t n_cap, const uint8_t* kI, const uint8_t* qI, const uint16_t* wI,
                            const uint16_t* q, const uint16_t* swa_ring, const float* sink, int32_t* idx_out,
                            uint16_t* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return layer_decode(p, B, q_pos, ring_Ca, ring_Za, ring_Cb, ring_Zb, Ba, Bb, rms_w, kv_comp, n_cap, kI, qI, wI, q,
                      swa_ring, sink, idx_out, out, lse, workspace, workspace_bytes, stream, nullptr);
}

csa_status csa_layer_decode_append(const csa_params* p, int32_t B, const int32_t* q_pos, const uint16_t* swa_new,
                                   const uint8_t* kI_new, const uint16_t* ring_Ca, const uint16_t* ring_Za,
                                   const uint16_t* ring_Cb, const uint16_t* ring_Zb, const uint16_t* Ba,
                                   const uint16_t* Bb, const uint16_t* rms_w, void* kv_comp, int64_t n_cap,
                                   uint8_t* kI, const uint8_t* qI, const uint16_t* wI, const uint16_t* q,
                                   uint16_t* swa_ring, const float* sink, int32_t* idx_out, uint16_t* out, float* lse,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if (!ok_ptr(swa_new) || !ok_opt(kI_new)) return CSA_ERR_INVALID_ARG;
  if (kI_new && p->index_format != 0) return CSA_ERR_UNSUPPORTED;  // E4M3 index keys only
  csa::DecodeAppend ap = {};
  ap.q_pos = q_pos;
  ap.B = B;
  ap.W = p->swa_window;
  ap.m = p->m;
  ap.swa_new = swa_new;
  ap.swa_ring = swa_ring;
  ap.kI_new = kI_new;
  ap.kI = kI;
  ap.n_cap = n_cap;
  return layer_decode(p, B, q_pos, ring_Ca, ring_Za, ring_Cb, ring_Zb, Ba, Bb, rms_w, kv_comp, n_cap, kI, qI, wI, q,
                      swa_ring, sink, idx_out, out, lse, workspace, workspace_bytes, stream, &ap);
}

csa_status csa_layer_decode_with_keys(const csa_params* p, int32_t B, const int32_t* q_pos, const uint16_t* swa_new,
                                      const csa_index_key_src* keys, const uint16_t* ring_Ca, const uint16_t* ring_Za,
                                      const uint16_t* ring_Cb, const uint16_t* ring_Zb, const uint16_t* Ba,
                                      const uint16_t* Bb, const uint16_t* rms_w, void* kv_comp, int64_t n_cap,
                                      uint8_t* kI, const uint8_t* qI, const uint16_t* wI, const uint16_t* q,
                                      uint16_t* swa_ring, const float* sink, int32_t* idx_out, uint16_t* out,
                                      float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if (!ok_opt(swa_new) || !key_src_ok(keys, false, 0)) return CSA_ERR_INVALID_ARG;
  if (p->index_format != 0) return CSA_ERR_UNSUPPORTED;  // E4M3 index keys only
  csa::DecodeAppend ap = {};
  ap.q_pos = q_pos;
  ap.B = B;
  ap.W = p->swa_window;
  ap.m = p->m;
  ap.swa_new = swa_new;
  ap.swa_ring = swa_ring;
  ap.kI = kI;
  ap.n_cap = n_cap;
  return layer_decode(p, B, q_pos, ring_Ca, ring_Za, ring_Cb, ring_Zb, Ba, Bb, rms_w, kv_comp, n_cap, kI, qI, wI, q,
                      swa_ring, sink, idx_out, out, lse, workspace, workspace_bytes, stream, &ap, keys, kI);
}

namespace {
// One prefill chunk; with `keys`, the compressor launch also writes the
// chunk's indexer keys into kI_out.
csa_status layer_prefill(const csa_params* p, int32_t B, int32_t Q, int64_t pos0, const uint16_t* Ca,
                             const uint16_t* Za, const uint16_t* Cb, const uint16_t* Zb, const uint16_t* Cb_prev,
                             const uint16_t* Zb_prev, const uint16_t* Ba, const uint16_t* Bb,
                             const uint16_t* rms_w, void* kv_comp, int64_t n_cap, const uint8_t* kI,
                             const uint8_t* qI, const uint16_t* wI, const uint16_t* q, const uint16_t* swa,
                             const float* sink, int32_t* idx_out, uint16_t* out, float* lse, void* workspace,
                             size_t workspace_bytes, void* stream, const csa_index_key_src* keys = nullptr,
                             uint8_t* kI_out = nullptr) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if ((s = check_overlapped(p)) != CSA_OK) return s;
  if (B < 0 || Q < 0 || B > 65535 || Q > 65535 || pos0 < 0 || pos0 % p->m != 0 || !n_cap_ok(n_cap))
    return CSA_ERR_INVALID_ARG;
  if (keys && (!key_src_ok(keys, true, pos0) || !ok_ptr(kI_out))) return CSA_ERR_INVALID_ARG;
  if (keys && p->index_format != 0) return CSA_ERR_UNSUPPORTED;
  if (B == 0 || Q == 0) return CSA_OK;
  const int64_t entry0 = pos0 / p->m;
  const int64_t n_new = (pos0 + Q) / p->m - entry0;
  if (entry0 + n_new > n_cap) return CSA_ERR_INVALID_ARG;
  if (!ok_ptr(Ca) || !ok_ptr(Za) || !ok_ptr(Cb) || !ok_ptr(Zb) || !ok_ptr(Ba) || !ok_ptr(Bb) || !ok_ptr(rms_w) ||
      !ok_ptr(kv_comp) || !ok_ptr(kI) || !ok_ptr(qI) || !ok_ptr(wI) || !ok_ptr(q) || !ok_ptr(swa) ||
      !ok_ptr(sink) || !ok_ptr(idx_out) || !ok_ptr(out) || !ok_opt(lse))
    return CSA_ERR_INVALID_ARG;
  if ((pos0 > 0) != (Cb_prev != nullptr) || (Cb_prev == nullptr) != (Zb_prev == nullptr) || !ok_opt(Cb_prev) ||
      !ok_opt(Zb_prev))
    return CSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  IndexWs w;
  if (!index_workspace(static_cast<int64_t>(B) * Q, n_cap, &w)) return CSA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return CSA_ERR_WORKSPACE;
  trace(0, st);
  if (csa::launch_zero(static_cast<uint8_t*>(workspace) + w.hist_off, w.zero_bytes, st) != cudaSuccess)
    return CSA_ERR_CUDA;
  uint16_t* kv16 = p->kv_format ? nullptr : static_cast<uint16_t*>(kv_comp);
  uint8_t* kv8 = p->kv_format ? static_cast<uint8_t*>(kv_comp) : nullptr;
  // 1. compress the chunk's complete blocks (and, with keys, their indexer
  //    keys in the same launch).  Rows are [B][Q][D]; the compressor reads
  //    m*n_new of them per sequence with a stride of Q rows.
  unsigned* status = status_ptr();
  if (!status) return CSA_ERR_CUDA;
  if (n_new > 0) {
    if (static_cast<int64_t>(Q) != n_new * p->m) {
      // Ragged chunk: compress sequence by sequence so the row stride is Q.
      for (int32_t b = 0; b < B; ++b) {
        const int64_t off = static_cast<int64_t>(b) * Q * csa::kDim;
        const int64_t poff = static_cast<int64_t>(b) * p->m * csa::kDim;
        csa::CompressArgs ka = {};
        if (keys) {
          const int64_t ko = static_cast<int64_t>(b) * Q * csa::kIdxDim, kp = static_cast<int64_t>(b) * p->m * csa::kIdxDim;
          csa_index_key_src kb = *keys;
          kb.CIa += ko, kb.ZIa += ko, kb.CIb += ko, kb.ZIb += ko;
          if (kb.CIb_prev) kb.CIb_prev += kp, kb.ZIb_prev += kp;
          ka = key_args(p, 0, 1, n_new, entry0, kb, kI_out + static_cast<int64_t>(b) * n_cap * csa::kIdxDim, n_cap,
                        nullptr, status);
        }
        s = run_compress(p, 0, 1, n_new, entry0, Ca + off, Za + off, Cb + off, Zb + off,
                         Cb_prev ? Cb_prev + poff : nullptr, Zb_prev ? Zb_prev + poff : nullptr, Ba, Bb, rms_w,
                         kv16 ? kv16 + static_cast<int64_t>(b) * n_cap * csa::kDim : nullptr, n_cap * csa::kDim, n_cap,
                         nullptr, st, kv8 ? kv8 + static_cast<int64_t>(b) * n_cap * csa::kFp4Entry : nullptr,
                         n_cap * csa::kFp4Entry, keys ? &ka : nullptr);
        if (s != CSA_OK) return s;
      }
    } else {
      csa::CompressArgs ka = {};
      if (keys) ka = key_args(p, 0, B, n_new, entry0, *keys, kI_out, n_cap, nullptr, status);
      s = run_compress(p, 0, B, n_new, entry0, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, rms_w, kv16,
                       n_cap * csa::kDim, n_cap, nullptr, st, kv8, n_cap * csa::kFp4Entry, keys ? &ka : nullptr);
      if (s != CSA_OK) return s;
    }
  }
  trace(1, st);
  // 2. indexer + top-k, each query over its own V(t)
  s = run_index_topk(p, B, Q, nullptr, pos0, qI, wI, kI, n_cap, idx_out, nullptr, workspace, workspace_bytes, st,
                     true, true);
  if (s != CSA_OK) return s;
  trace(3, st);
  // 3. sparse attention with the linear window (row j = position pos0-(W-1)+j)
  const size_t attn_off = round_up(w.total, 256);
  s = run_attn(p, B, Q, nullptr, pos0, q, kv_comp, n_cap, idx_out, swa, 1, static_cast<int64_t>(p->swa_window) - 1 + Q,
               nullptr, pos0 - (p->swa_window - 1), sink, out, lse, st, false,
               static_cast<uint8_t*>(workspace) + attn_off, workspace_bytes > attn_off ? workspace_bytes - attn_off : 0);
  trace(4, st);
  return s;
}
}  // namespace

csa_status csa_layer_prefill(const csa_params* p, int32_t B, int32_t Q, int64_t pos0, const uint16_t* Ca,
                             const uint16_t* Za, const uint16_t* Cb, const uint16_t* Zb, const uint16_t* Cb_prev,
                             const uint16_t* Zb_prev, const uint16_t* Ba, const uint16_t* Bb,
                             const uint16_t* rms_w, void* kv_comp, int64_t n_cap, const uint8_t* kI,
                             const uint8_t* qI, const uint16_t* wI, const uint16_t* q, const uint16_t* swa,
                             const float* sink, int32_t* idx_out, uint16_t* out, float* lse, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return layer_prefill(p, B, Q, pos0, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, rms_w, kv_comp, n_cap, kI, qI, wI, q,
                       swa, sink, idx_out, out, lse, workspace, workspace_bytes, stream);
}

csa_status csa_layer_prefill_with_keys(const csa_params* p, int32_t B, int32_t Q, int64_t pos0, const uint16_t* Ca,
                                       const uint16_t* Za, const uint16_t* Cb, const uint16_t* Zb,
                                       const uint16_t* Cb_prev, const uint16_t* Zb_prev, const uint16_t* Ba,
                                       const uint16_t* Bb, const uint16_t* rms_w, const csa_index_key_src* keys,
                                       void* kv_comp, int64_t n_cap, uint8_t* kI, const uint8_t* qI,
                                       const uint16_t* wI, const uint16_t* q, const uint16_t* swa, const float* sink,
                                       int32_t* idx_out, uint16_t* out, float* lse, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  if (!keys) return CSA_ERR_INVALID_ARG;
  return layer_prefill(p, B, Q, pos0, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, rms_w, kv_comp, n_cap, kI, qI, wI, q,
                       swa, sink, idx_out, out, lse, workspace, workspace_bytes, stream, keys, kI);
}

csa_status csa_hca_layer_decode(const csa_params* p, int32_t B, const int32_t* q_pos, const uint16_t* C,
                                const uint16_t* Z, const uint16_t* bias, const uint16_t* rms_w, float* state,
                                uint16_t* kv_comp, int64_t n_cap, const uint16_t* q, const uint16_t* swa_ring,
                                const float* sink, uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                                void* stream) {
  csa_status s = check_params(p);
  if (s != CSA_OK) return s;
  if ((s = check_bf16_cache(p)) != CSA_OK) return s;
  if (B < 0 || B > 65535 || !n_cap_ok(n_cap)) return CSA_ERR_INVALID_ARG;
  if (B == 0) return CSA_OK;
  if (!ok_ptr(q_pos) || !ok_ptr(C) || !ok_ptr(Z) || !ok_opt(bias) || !ok_ptr(rms_w) || !ok_ptr(state) ||
      !ok_ptr(kv_comp) || !ok_ptr(q) || !ok_ptr(swa_ring) || !ok_ptr(sink) || !ok_ptr(out) || !ok_opt(lse))
    return CSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = status_ptr();
  if (!status) return CSA_ERR_CUDA;
  trace(0, st);
  // 1. the step's token into the compressor state; a completed block's entry into the cache
  csa::CompressArgs ca = compress_args(p, 1, B, 0, 0, C, Z, nullptr, nullptr, nullptr, nullptr, bias, nullptr, rms_w,
                                       kv_comp, n_cap * csa::kDim, n_cap, q_pos, status);
  ca.state = state;
  if ((s = cuda_status(csa::launch_compress_single(ca, st))) != CSA_OK) return s;
  trace(1, st);
  trace(2, st);
  trace(3, st);
  // 2. dense attention: the ring window and every visible entry (the new one included)
  s = run_attn(p, B, 1, q_pos, 0, q, kv_comp, n_cap, nullptr, swa_ring, 0, p->swa_window, nullptr, 0, sink, out, lse,
               st, true, workspace, workspace_bytes);
  trace(4, st);
  return s;
}

uint64_t csa_launch_count(void) { return csa::g_launches.load(std::memory_order_relaxed); }

csa_status csa_set_trace_events(void* const* events, int32_t n_events) {
  if (!events) {
    g_trace_on = false;
    return CSA_OK;
  }
  if (n_events != 5) return CSA_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i) {
    if (!events[i]) return CSA_ERR_INVALID_ARG;
    g_trace[i] = static_cast<cudaEvent_t>(events[i]);
  }
  g_trace_on = true;
  return CSA_OK;
}

csa_status csa_test_set_wait_fault(uint32_t wait_limit_us, uint32_t faults) {
  if (faults & ~(CSA_TEST_FAULT_INDEXER | CSA_TEST_FAULT_TOPK | CSA_TEST_FAULT_ATTN)) return CSA_ERR_INVALID_ARG;
  if (faults && wait_limit_us == 0) return CSA_ERR_INVALID_ARG;  // a fault waits out the test limit only
  unsigned* p = status_ptr();
  if (!p) return CSA_ERR_CUDA;
  static_assert(CSA_TEST_FAULT_INDEXER == csa::kFaultIndexer && CSA_TEST_FAULT_TOPK == csa::kFaultTopk &&
                    CSA_TEST_FAULT_ATTN == csa::kFaultAttn,
                "fault bits");
  const unsigned words[2] = {faults, wait_limit_us};
  if (cudaDeviceSynchronize() != cudaSuccess) return CSA_ERR_CUDA;  // no kernel reads them meanwhile
  return cudaMemcpy(p + 1, words, sizeof words, cudaMemcpyHostToDevice) == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

csa_status csa_check_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return CSA_ERR_CUDA;
  unsigned* p = status_ptr();
  if (!p) return CSA_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, p, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
  const unsigned zero = 0;
  if (word && cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return CSA_ERR_CUDA;
  if (word & csa::kErrTimeout) return CSA_ERR_TIMEOUT;
  if (word & csa::kErrIndexRange) return CSA_ERR_INDEX_RANGE;
  return CSA_OK;
}

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_INVALID_ARG: return "CSA_ERR_INVALID_ARG: null, misaligned or out-of-range argument";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED: dimensions other than the supported CSA shape";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA: a CUDA call or launch failed";
    case CSA_ERR_TIMEOUT: return "CSA_ERR_TIMEOUT: a bounded device-side wait gave up";
    case CSA_ERR_INDEX_RANGE: return "CSA_ERR_INDEX_RANGE: a position or index pointed outside a cache";
    case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE: workspace missing or too small";
  }
  return "CSA_ERR_UNKNOWN";
}

}  // extern "C"
