/*
 * libcsa — the hot path of one Compressed Sparse Attention (CSA) layer on
 * NVIDIA GB300 (sm_103a): compressor, lightning indexer + top-k, and the
 * shared-KV sparse MQA with an attention sink, for decode and chunked prefill.
 *
 * Page titles used in the citations below:
 *   [hca_csa]   "CSA / HCA" (zdszero.github.io, hca_csa)
 *   [KV 压缩]   "DeepSeek-V4 的 KV 压缩：从删 token 误解到预算检索"
 *   [CSA2 详解] "DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2：从模型原理到推理基础设施"
 *   [结构对比]  "DeepSeek 注意力结构对比：MHA、GQA、MLA、DSA、CSA、HCA、CSA2"
 *   [CED]       "从 GPT 到 CED：DeepSeek-V4.1-Flash 如何改变上下文的计算方式"
 *
 * Conventions shared by every call
 * --------------------------------
 * - Plain C ABI.  bf16 tensors are passed as `uint16_t*` (raw bfloat16 bits),
 *   FP8 E4M3 (finite-only "fn" variant, no scale) as `uint8_t*`.
 * - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *   never allocates device memory.  Scratch memory ("workspace") is passed by
 *   the caller and must be at least csa_workspace_size() bytes.
 * - `stream` is a cudaStream_t passed as `void*` (NULL = legacy default stream).
 *   Every call is asynchronous on that stream.
 * - Layouts are dense row-major unless a stride argument says otherwise.  All
 *   base pointers must be 16-byte aligned.
 * - Argument errors are detected on the host before any launch and returned
 *   (CSA_ERR_INVALID_ARG / CSA_ERR_UNSUPPORTED / CSA_ERR_WORKSPACE); outputs
 *   are then left untouched.  A failed launch returns CSA_ERR_CUDA.
 * - Data-dependent errors (a position or index outside the caches, a bounded
 *   device-side wait that gave up) cannot be seen by the host at call time.
 *   The kernels clamp the offending access, keep running, and record the
 *   error in a device status word; csa_check_status() reports and clears it.
 *   No kernel traps.
 * - The model dimensions are fixed by the pages for V4-Flash/Pro CSA layers
 *   ([CSA2 详解] §3.1; [hca_csa] "CSA：轻压缩 + 稀疏选择"): 64 query heads of
 *   width 512 sharing one 512-wide K=V latent, partial RoPE on its last 64
 *   channels, 64 indexer heads of width 128.  Calls with other values return
 *   CSA_ERR_UNSUPPORTED.
 */
#ifndef LIBCSA_CSA_H
#define LIBCSA_CSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer     */
  CSA_ERR_UNSUPPORTED = 2,  /* a dimension other than the ones listed above   */
  CSA_ERR_CUDA = 3,         /* a CUDA runtime call or a launch failed         */
  CSA_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up             */
  CSA_ERR_INDEX_RANGE = 5,  /* a position / index pointed outside a cache     */
  CSA_ERR_WORKSPACE = 6     /* workspace missing or smaller than required     */
} csa_status;

/* Hyper-parameters of one CSA layer. */
typedef struct {
  int32_t m;          /* compression ratio: one entry per m tokens (4); a
                         power of two, 1..8 for the overlapped CSA compressor
                         and the layer calls, up to 128 for the single-stream
                         compressor and dense attention (HCA: 128)          */
  int32_t n_heads;    /* query heads (64)                                    */
  int32_t head_dim;   /* shared K=V latent width (512)                        */
  int32_t rope_dim;   /* trailing channels that carry RoPE (64)               */
  int32_t idx_heads;  /* lightning-indexer heads n_h^I (64)                   */
  int32_t idx_dim;    /* lightning-indexer width c^I (128)                    */
  int32_t topk;       /* entries selected per query, 1..2048 (512 or 1024)    */
  int32_t swa_window; /* raw sliding-window rows per query, 1..1024 (128)     */
  float rope_theta;   /* RoPE base (1e4)                                      */
  float rms_eps;      /* RMSNorm epsilon (1e-6)                               */
  float sm_scale;     /* logit scale applied to q·kv (1/sqrt(512))            */
  int32_t inverse_rope; /* 1: rotate the output's last rope_dim channels back
                           by the query position (see csa_sparse_attn); 0    */
  int32_t kv_format;  /* compressed cache entries: 0 bf16 (512 x 2 B), 1 FP4
                         (CSA_FP4_ENTRY_BYTES, see csa_quantize_kv_fp4).
                         csa_layer_decode(_append) / csa_layer_prefill read
                         and write their kv_comp in this format (the compressor
                         stores the FP4 entry of its bf16 values);
                         csa_compress and the single-stream calls write
                         bf16 only                                       */
  int32_t bf16_scores; /* 1: the indexer rounds each score to bf16 (nearest,
                           ties to even) and the top-k selects on the rounded
                           values, ties to the smaller entry as always;
                           score_out returns the rounded values.  Halves the
                           score traffic ([KV 压缩] §7, "Oracle top-k vs
                           learned top-k": BF16 scores for the selector).
                           0: fp32 scores                                 */
  int32_t index_format; /* the indexer's keys kI and queries qI: 0 E4M3
                           codes (kI [B][n_cap][128], qI [B][Q][64][128]);
                           1 FP4 (E2M1 codes, one E8M0 scale per 32 values,
                           the layouts of csa_quantize_index_keys_fp4 and
                           csa_quantize_index_query_fp4)                  */
} csa_params;

#define CSA_FP4_ENTRY_BYTES 288

/* Fills *p with the V4-Flash CSA values listed above (topk = 512). */
void csa_default_params(csa_params *p);

/* Operation codes for csa_workspace_size(). */
enum {
  CSA_OP_COMPRESS = 0,
  CSA_OP_INDEX_TOPK = 1,
  CSA_OP_SPARSE_ATTN = 2,
  CSA_OP_LAYER_DECODE = 3,
  CSA_OP_LAYER_PREFILL = 4,
  CSA_OP_INDEX_TOPK_POOL = 5,
  CSA_OP_REINDEX_TOPK = 6,
  CSA_OP_HCA_LAYER_DECODE = 7
};

/* Bytes of workspace the call `op` needs for B sequences of Q queries over a
 * cache of n_cap entries.  Returns 0 for an invalid combination.  The
 * attention's share (CSA_OP_SPARSE_ATTN and the layer calls) is sized for
 * the current device: one wave of split-KV slices, min(16, SMs / (B*Q))
 * per query, none when fewer than 2 fit. */
size_t csa_workspace_size(int32_t op, const csa_params *p, int32_t B, int32_t Q,
                          int64_t n_cap);

/*
 * csa_compress — overlapped compressor, bulk form.
 * [hca_csa] "CSA 的重叠窗口", the Softmax_row and C_i^Comp equations, and
 * "压缩算子：逐通道 softmax 的软池化"; i = 0 boundary in the same section;
 * RoPE position = first token of the entry's own block ([CSA2 详解] §7.4).
 *
 * For every sequence b and every entry i in [entry0, entry0 + n_new):
 *   per channel d, softmax over the 2m logits
 *     Za[b, m*i + r, d] + Ba[r, d]            (block i, slots r = 0..m-1)
 *     Zb[b, m*(i-1) + r, d] + Bb[r, d]        (block i-1)
 *   weights the matching rows of Ca / Cb and sums them; the 512-vector is then
 *   RMS-normalised (eps = p->rms_eps) and scaled by rms_w, and the last
 *   rope_dim channels are rotated in interleaved pairs (D-R+2j, D-R+2j+1) by
 *   angle (m*i) * rope_theta^(-2j/R).  For i = 0 the block-(i-1) slots are
 *   absent (logit -inf, value 0).
 *
 * Ca, Za, Cb, Zb : [B][m*n_new][D] bf16 — rows of the chunk's tokens; row j of
 *                  sequence b is token m*entry0 + j.
 * Cb_prev, Zb_prev: [B][m][D] bf16 — Cb/Zb rows of the m tokens before the
 *                  chunk (block entry0-1).  Must be NULL iff entry0 == 0.
 * Ba, Bb         : [m][D] bf16 block-slot biases ("ape").
 * rms_w          : [D] bf16 RMSNorm weight.
 * kv_out         : entry e of sequence b is written at
 *                  kv_out + b*kv_stride_b + e*D (bf16); rows entry0.. only.
 */
csa_status csa_compress(const csa_params *p, int32_t B, int32_t n_new,
                        int64_t entry0, const uint16_t *Ca, const uint16_t *Za,
                        const uint16_t *Cb, const uint16_t *Zb,
                        const uint16_t *Cb_prev, const uint16_t *Zb_prev,
                        const uint16_t *Ba, const uint16_t *Bb,
                        const uint16_t *rms_w, uint16_t *kv_out,
                        int64_t kv_stride_b, void *stream);

/*
 * csa_compress_indexer_keys — the lightning indexer's own key compressor,
 * bulk form.  [hca_csa] "CSA：轻压缩 + 稀疏选择": the indexer keeps a
 * compressed K of its own (head_dim 128, one entry per m tokens at the same
 * entry numbering as the main cache), rotated by a Hadamard matrix after
 * compression so that it quantises well to FP8.
 *
 * For every sequence b and entry i in [entry0, entry0 + n_new): the steps of
 * csa_compress at width 128 (the 2m-slot softmax pooling of CIa/CIb by the
 * logits ZIa+BIa / ZIb+BIb, RMSNorm with rms_wI and eps = p->rms_eps, RoPE
 * on the last rope_dim channels in interleaved pairs at position m*i), then
 * y = H_128 x / sqrt(128) with H the Sylvester Hadamard matrix (entry (r, c)
 * = (-1)^popcount(r & c)), then each y_d stored as the nearest FP8 E4M3 code
 * (ties to the even code, magnitudes past 448 saturate to +-448, no scale).
 *
 * CIa, ZIa, CIb, ZIb : [B][m*n_new][128] bf16, row j of sequence b is token
 *                      m*entry0 + j.
 * CIb_prev, ZIb_prev : [B][m][128] bf16 rows of block entry0-1, NULL iff
 *                      entry0 == 0.
 * BIa, BIb : [m][128] bf16.   rms_wI : [128] bf16.
 * kI_out   : entry e of sequence b at kI_out + b*kI_stride_b + e*128 (E4M3
 *            bytes, the layout csa_index_topk reads); rows entry0.. only.
 */
csa_status csa_compress_indexer_keys(
    const csa_params *p, int32_t B, int32_t n_new, int64_t entry0,
    const uint16_t *CIa, const uint16_t *ZIa, const uint16_t *CIb,
    const uint16_t *ZIb, const uint16_t *CIb_prev, const uint16_t *ZIb_prev,
    const uint16_t *BIa, const uint16_t *BIb, const uint16_t *rms_wI,
    uint8_t *kI_out, int64_t kI_stride_b, void *stream);

/*
 * csa_compress_single — the non-overlapped compressor of HCA and CSA2 layers,
 * bulk form.  [hca_csa] "HCA：同一个算子，关掉重叠" (one stream C, Z and
 * slot bias B, Softmax_row over the m slots of the entry's own block);
 * [CSA2 详解] §7.2 (CSA2: the same pooling without the slot bias) and §7.5
 * (m = 1: the softmax weight is 1, the entry is RoPE(Norm(C))).  m = p->m,
 * a power of two up to 128 (HCA uses 128).
 *
 * For every sequence b and entry i in [entry0, entry0 + n_new), per channel
 * d: softmax over the m logits Z[b, m*(i-entry0) + r, d] + bias[r, d]
 * (bias NULL: no bias) weighting the rows C[b, m*(i-entry0) + r, :]; then
 * RMSNorm (p->rms_eps) times rms_w and RoPE on the last 64 channels in
 * interleaved pairs at position m*i, as csa_compress does.
 *
 * C, Z   : [B][m*n_new][512] bf16, row j of sequence b is token m*entry0 + j.
 * bias   : [m][512] bf16 or NULL.          rms_w : [512] bf16.
 * kv_out : entry e of sequence b at kv_out + b*kv_stride_b + e*512 (bf16).
 * m above 128 or not a power of two: CSA_ERR_UNSUPPORTED.
 */
csa_status csa_compress_single(const csa_params *p, int32_t B, int32_t n_new,
                               int64_t entry0, const uint16_t *C,
                               const uint16_t *Z, const uint16_t *bias,
                               const uint16_t *rms_w, uint16_t *kv_out,
                               int64_t kv_stride_b, void *stream);

/*
 * csa_compress_single_step — the same compressor at decode, one token per
 * sequence per call, with an online softmax: per channel the block's tokens
 * so far are held as a running (max logit, sum of e^(logit - max), sum of
 * e^(logit - max) * C) instead of their rows ([hca_csa] "KV cache：成品与
 * 原料": the HCA compressor's state shrinks to one (max, sum, kv) slot).
 *
 * For each b with t = q_pos[b] >= 0 and slot r = t mod m: the token's logit
 * Z[b,:] + bias[r,:] and row C[b,:] start the state (r == 0) or are folded
 * into it; when r == m-1 the block is complete and entry i = (t+1)/m - 1 is
 * written to kv_out + b*kv_stride_b + i*512 (RMSNorm, RoPE at m*i); an i at
 * or past n_cap records CSA_ERR_INDEX_RANGE.  The result equals
 * csa_compress_single over the same block up to fp32 rounding.
 *
 * C, Z  : [B][512] bf16, this step's token.      bias : [m][512] or NULL.
 * state : [B][3][512] fp32, owned by the caller, read and written by every
 *         call; a sequence must be stepped through its positions in order
 *         (its state is valid only after the first token of a block).
 */
csa_status csa_compress_single_step(const csa_params *p, int32_t B,
                                    const int32_t *q_pos, const uint16_t *C,
                                    const uint16_t *Z, const uint16_t *bias,
                                    const uint16_t *rms_w, float *state,
                                    uint16_t *kv_out, int64_t kv_stride_b,
                                    int64_t n_cap, void *stream);

/*
 * csa_index_topk — lightning indexer + top-k over the causally visible entries.
 * Score: [hca_csa] "CSA：轻压缩 + 稀疏选择", equation I_{t,s}; also
 * [结构对比] DSA section.  Visibility: [KV 压缩] §9.8 (entry s is visible to
 * the query at position t iff (s+1)*m <= t+1, i.e. s < V(t) = floor((t+1)/m)).
 * Selection over all visible entries, window included ([hca_csa] "top-k 的选择
 * 范围不排除 SWA 窗口").
 *
 *   I[b,q,s] = sum_h wI[b,q,h] * max(0, sum_c qI[b,q,h,c] * kI[b,s,c])
 *
 * for s < V(q_pos[b,q]); the min(topk, V) entries with the largest I are
 * returned in idx_out[b,q,:] in ascending entry order, followed by -1 for the
 * remaining slots.  Equal scores are broken toward the smaller entry index.
 * score_out (optional) receives the fp32 score of each returned entry (and
 * -inf in the -1 slots).
 *
 * q_pos : [B][Q] int32, absolute token position of each query.  V(t) must not
 *         exceed n_cap (else CSA_ERR_INDEX_RANGE is recorded and V is clamped).
 * qI    : [B][Q][64][128] e4m3.      wI : [B][Q][64] bf16 (scale included).
 * kI    : [B][n_cap][128] e4m3 indexer keys, entry numbering shared with the
 *         main compressed KV (one indexer key per compressed entry, [hca_csa]).
 * idx_out: [B][Q][topk] int32.  score_out: [B][Q][topk] fp32 or NULL.
 * Accuracy: FP8 products are exact; they are accumulated in fp32 by the tensor
 * cores and the head sum is fp32.
 */
csa_status csa_index_topk(const csa_params *p, int32_t B, int32_t Q,
                          const int32_t *q_pos, const uint8_t *qI,
                          const uint16_t *wI, const uint8_t *kI, int64_t n_cap,
                          int32_t *idx_out, float *score_out, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * csa_index_topk_static — csa_index_topk without a caller-provided workspace.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory where they call the indexer: for example a
 * serving process whose own pool allocator has reserved the GPU's memory up
 * front (a cudaMalloc would fail or take memory the pool counts on), or a
 * latency-critical loop that must not call cudaMalloc because it can block
 * the host and synchronise the device.
 *
 * Arguments, results and errors are those of csa_index_topk.  The scratch is
 * one fixed device array inside libcsa of CSA_STATIC_SCRATCH_BYTES (16 MiB)
 * that every GPU that loads the library holds until the process exits; a call
 * whose scratch need, csa_workspace_size(CSA_OP_INDEX_TOPK, ...), exceeds it
 * returns CSA_ERR_WORKSPACE without launching anything.  The call allocates
 * nothing.  The first call on each device (with that device current) looks
 * up the array's device address; make that first call before any stream
 * capture.  Every call uses the same array, which keeps the previous call's
 * contents (nothing in it needs to start at zero): calls that can run on the
 * GPU at the same time (other streams, other host threads) race on it, so
 * the caller must serialise them.
 */
#define CSA_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
csa_status csa_index_topk_static(const csa_params *p, int32_t B, int32_t Q,
                                 const int32_t *q_pos, const uint8_t *qI,
                                 const uint16_t *wI, const uint8_t *kI,
                                 int64_t n_cap, int32_t *idx_out,
                                 float *score_out, void *stream);

/*
 * csa_quantize_kv_fp4 — compressed cache entries to the FP4 layout ([CSA2 详解]
 * §16.1: 512 FP4 values and one 1-byte E4M3 scale per 16 values, 288 bytes).
 * Entry layout: bytes 0..255 the E2M1 codes, channel 2j in the low nibble of
 * byte j and 2j+1 in the high nibble; bytes 256..287 the E4M3 scales, scale g
 * for channels 16g..16g+15.  Scale of a group: the E4M3 code nearest to
 * amax/6 (amax its largest magnitude); code of a channel: the E2M1 code
 * nearest to x/scale (ties to the even code, saturating at +-6, the sign
 * kept); both quotients are formed in binary32; a zero scale gives zero
 * codes.  The entry stands for scale * e2m1(code).
 *
 * in  : n_rows rows of 512 bf16, row r at in + r*in_stride (elements).
 * out : entry r at out + r*out_stride (bytes, a multiple of 16, >= 288).
 */
csa_status csa_quantize_kv_fp4(int64_t n_rows, const uint16_t *in,
                               int64_t in_stride, uint8_t *out,
                               int64_t out_stride, void *stream);

/*
 * FP4 indexer keys and queries ([CSA2 详解] §16.2 "一份 Indexer K": a key of
 * 128 FP4 values and one 1-byte E8M0 scale per 32 values, 68 bytes; the
 * indexer's query is FP4 too, [结构对比] CSA2 figure; [KV 压缩] §7.2 "Oracle
 * top-k vs learned top-k": the CSA indexer's QK path in FP4).  A block of 32
 * values with largest magnitude amax gets the scale s = 2^e, e the smallest
 * integer in -127..127 with 6 * 2^e >= amax (the pages leave the rounding
 * open; this one keeps every x/s within E2M1's range, so no code saturates);
 * each value x gets the E2M1 code nearest to x/s (the quotient is exact; ties
 * to the even code; the sign is kept, so a small negative value gives -0).
 * The value stands for s * e2m1(code).  Inputs must be finite.
 *
 * Key cache of B sequences of n_cap entries (CSA_FP4_INDEX_KEYS_BYTES bytes):
 *   codes  : entry e of sequence b at kI + (b*n_cap + e)*64; byte j holds
 *            channel 2j in its low nibble and 2j+1 in its high nibble.
 *   scales : after all codes, 512 bytes per 128 entries of each sequence:
 *            the scale of channels 32g..32g+31 of entry e of sequence b at
 *            kI + B*n_cap*64 + b*512*ceil(n_cap/128) + 512*(e/128)
 *               + 16*(e%32) + 4*((e%128)/32) + g
 *            (the order in which the tensor cores read them).
 * Query records, one per query, n_q = B*Q of them (CSA_FP4_INDEX_QUERY_BYTES):
 *   codes  : head h of query r at qI + (64*r + h)*64, same nibble order.
 *   scales : after all codes, 512 bytes per query: block g of head h of
 *            query r at qI + n_q*4096 + 512*r + 16*(h%32) + 4*(h/32) + g;
 *            bytes 8..15 of every 16-byte line are zero.
 */
#define CSA_FP4_INDEX_KEYS_BYTES(B, n_cap) \
  ((size_t)(B) * ((size_t)(n_cap) * 64u + (((size_t)(n_cap) + 127u) / 128u) * 512u))
#define CSA_FP4_INDEX_QUERY_BYTES(n_q) ((size_t)(n_q) * 4608u)

/*
 * csa_quantize_index_keys_fp4 — bf16 indexer keys into the FP4 key cache.
 * in : row j (128 bf16) of sequence b at in + b*in_stride_b + j*128 for
 *      j < n_new (in_stride_b a multiple of 8 and >= n_new*128 when B > 1).
 * kI : the FP4 key cache (B sequences of n_cap entries, layout above);
 *      entries entry0 .. entry0+n_new-1 are written (entry0 + n_new <=
 *      n_cap), all others are left as they are.
 * Device pointers, 16-byte aligned.  No workspace.
 */
csa_status csa_quantize_index_keys_fp4(int32_t B, int32_t n_new,
                                       int64_t entry0, const uint16_t *in,
                                       int64_t in_stride_b, uint8_t *kI,
                                       int64_t n_cap, void *stream);

/*
 * csa_quantize_index_query_fp4 — bf16 indexer queries [n_q][64][128] (n_q =
 * B*Q, contiguous) into n_q FP4 query records at qI (layout above).
 */
csa_status csa_quantize_index_query_fp4(int64_t n_q, const uint16_t *in,
                                        uint8_t *qI, void *stream);

/*
 * Hierarchical indexer ([CSA2 详解] §11 "Hierarchical Sparse Indexer"; §11.1
 * on why the pool is larger than top-k; §20.1: a Reindex layer gathers the
 * candidates before it scores them).  A Full layer scores every visible
 * entry, keeps its own top-k, and hands on a candidate pool: entries grouped
 * in blocks of CSA_POOL_BLOCK consecutive ones, a block scored by the largest
 * score among its visible entries, the pool_blocks best blocks kept.  A
 * Reindex layer scores only the pool's entries, with its own qI and wI, and
 * takes its own top-k among them.
 *
 * csa_index_topk_pool — a Full layer: everything csa_index_topk does, plus
 *   pool_out[b,q,:] = the min(pool_blocks, ceil(V/8)) block ids j (block j =
 *   entries 8j .. 8j+7, those below V(t) counted) with the largest block
 *   scores max_{s in block j, s < V} I[b,q,s], in ascending order, then -1.
 *   Equal block scores: the smaller block id first.
 *   pool_blocks : 16..2048, a multiple of 16 (the pages use 2048: at most
 *                 16384 candidates).
 *   pool_out    : [B][Q][pool_blocks] int32.
 *   Workspace   : csa_workspace_size(CSA_OP_INDEX_TOPK_POOL, p, B, Q, n_cap).
 *
 * csa_reindex_topk — a Reindex layer over the pool a Full layer made for the
 *   same q_pos (same B, Q, n_cap and pool_blocks):
 *     I[b,q,s] = sum_h wI[b,q,h] * max(0, sum_c qI[b,q,h,c] * kI[b,s,c])
 *   for the entries s of the pool's blocks with s < V(t) only; idx_out[b,q,:]
 *   receives the min(topk, #pool entries) entries with the largest I in
 *   ascending entry order (equal scores: the smaller entry), then -1;
 *   score_out (optional) their fp32 scores, -inf in the -1 slots.  The key
 *   rows read are those of the pool's blocks (1 KiB each, 16 per tensor-core
 *   tile), so the cost is fixed by pool_blocks, not by V.
 *   pool        : [B][Q][pool_blocks] int32 as csa_index_topk_pool wrote it.
 *                 A pool from other inputs gives unspecified selections but
 *                 no access outside kI (block ids past the cache record
 *                 CSA_ERR_INDEX_RANGE and are not scored).
 *   Workspace   : csa_workspace_size(CSA_OP_REINDEX_TOPK, p, B, Q, n_cap)
 *                 (sized for pool_blocks = 2048).
 *
 * Other arguments, layouts, accuracy and errors are those of csa_index_topk.
 * pool_blocks outside its range returns CSA_ERR_UNSUPPORTED.
 */
#define CSA_POOL_BLOCK 8
csa_status csa_index_topk_pool(const csa_params *p, int32_t B, int32_t Q,
                               const int32_t *q_pos, const uint8_t *qI,
                               const uint16_t *wI, const uint8_t *kI,
                               int64_t n_cap, int32_t *idx_out,
                               float *score_out, int32_t pool_blocks,
                               int32_t *pool_out, void *workspace,
                               size_t workspace_bytes, void *stream);
csa_status csa_reindex_topk(const csa_params *p, int32_t B, int32_t Q,
                            const int32_t *q_pos, const uint8_t *qI,
                            const uint16_t *wI, const uint8_t *kI,
                            int64_t n_cap, const int32_t *pool,
                            int32_t pool_blocks, int32_t *idx_out,
                            float *score_out, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * csa_sparse_attn — shared-KV MQA over [SWA rows || selected entries || sink].
 * [hca_csa] "设计：近处看原文，远处看摘要", the o_{t,i} equation and the bullet
 * on attn_sink; gather semantics [KV 压缩] §9.6; window [KV 压缩] §9.5.
 *
 * For the query at position t (= q_pos[b,q]) and head h, the row set is
 *   the raw window rows of positions max(0, t-W+1) .. t   (W = swa_window)
 *   the compressed rows kv_comp[b, idx[b,q,j]] for every idx != -1,
 * l_{h,j} = sm_scale * q[b,q,h,:] . row_j, and
 *   out[b,q,h,:] = sum_j e^{l_hj} row_j / (sum_j e^{l_hj} + e^{sink[h]}).
 * The sink enters the denominator only and is not scaled by sm_scale.
 * lse[b,q,h] (optional) = log(sum_j e^{l_hj} + e^{sink[h]}).
 *
 * q      : [B][Q][64][512] bf16.
 * kv_comp: p->kv_format 0: [B][n_cap][512] bf16; 1: [B][n_cap][288] FP4
 *          entries (csa_quantize_kv_fp4), gathered at 288 B per row and
 *          expanded to bf16 on chip (value * scale is exact in bf16).  The
 *          window rows are bf16 either way.
 * idx    : [B][Q][topk] int32, -1 marks an empty slot; any other value outside
 *          [0, n_cap) records CSA_ERR_INDEX_RANGE and the slot is skipped.
 *          NULL: dense attention, the HCA read path ([hca_csa] "HCA：同一个
 *          算子，关掉重叠"; [CSA2 详解] §9: a layer without an indexer reads
 *          every causally visible compressed entry): the compressed rows are
 *          kv_comp[b, 0 .. V(t)-1] with V(t) = floor((t+1)/p->m) (a V(t) past
 *          n_cap records CSA_ERR_INDEX_RANGE and is clamped).
 * swa    : swa_mode 0 (decode ring): [B][W][512], position u in slot u mod W.
 *          swa_mode 1 (linear):      [B][swa_len][512], row j holds position
 *          swa_pos0[b] + j (swa_pos0 is a [B] int32 device array); a needed
 *          position outside the buffer records CSA_ERR_INDEX_RANGE and is
 *          skipped.
 * sink   : [64] fp32.   out : [B][Q][64][512] bf16.   lse : [B][Q][64] or NULL.
 *
 * workspace: optional.  With csa_workspace_size(CSA_OP_SPARSE_ATTN, p, B, Q,
 *          n_cap) bytes (a token amount when B*Q > SMs/2), each query's rows
 *          may be cut into as many slices as the workspace holds and one
 *          wave of CTAs allows (up to 16, at most one per 128 rows), one CTA
 *          each, merged by a second kernel (the same result up to fp32
 *          summation order): taken when that gives more slices than a
 *          thread-block cluster holds, or slices of at most 3 tiles of 128
 *          rows.  Otherwise (and with NULL or too few bytes): one launch, at
 *          most a thread-block cluster's slices per query, merged on chip.
 *
 * With p->inverse_rope = 1 each head's output then gets the inverse of the
 * RoPE the rows carry, at the query position ([CSA2 详解] §12.1 "Partial RoPE
 * 与 inverse RoPE"; [KV 压缩] §9.6 kernel note): channels (448+2j, 449+2j)
 * are rotated by the angle -t * rope_theta^(-2j/64), the same interleaved
 * pairing and frequencies as the compressor's RoPE.  The layer calls pass
 * the flag through.  Any value other than 0 or 1 is CSA_ERR_INVALID_ARG.
 */
csa_status csa_sparse_attn(const csa_params *p, int32_t B, int32_t Q,
                           const int32_t *q_pos, const uint16_t *q,
                           const void *kv_comp, int64_t n_cap,
                           const int32_t *idx, const uint16_t *swa,
                           int32_t swa_mode, int64_t swa_len,
                           const int32_t *swa_pos0, const float *sink,
                           uint16_t *out, float *lse, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * csa_layer_decode — one decode step of a CSA layer for B sequences (Q = 1).
 * Order of the path: [KV 压缩] §9.9; emission at block boundaries [KV 压缩]
 * §9.3 and [hca_csa] "KV cache：成品与原料" (an entry is produced only when
 * (t+1) mod m == 0, reading the 2m staged rows).
 *
 *   1. if (q_pos[b]+1) % m == 0: entry i = (q_pos[b]+1)/m - 1 is compressed
 *      from the staged rows (block i from ring_Ca/Za, block i-1 from
 *      ring_Cb/Zb) and written to kv_comp[b, i];
 *   2. csa_index_topk over the V(t) visible entries;
 *   3. csa_sparse_attn with the ring window (swa_mode 0).
 *
 * ring_Ca/Za/Cb/Zb: [B][2m][512] bf16 compressor staging rows; the row of
 *         token u sits in slot u mod 2m and the slots hold tokens t-2m+1..t.
 * kI    : [B][n_cap][128] e4m3 — must already hold entries 0..V(t)-1 (the
 *         indexer keys come from a separate compressor that is not part of
 *         this call; csa_layer_decode_with_keys computes the step's key).
 * swa_ring: [B][W][512] bf16 holding positions t-W+1..t (slot u mod W).
 * idx_out: [B][topk] int32 (the selection), out [B][64][512], lse [B][64] or NULL.
 */
csa_status csa_layer_decode(
    const csa_params *p, int32_t B, const int32_t *q_pos,
    const uint16_t *ring_Ca, const uint16_t *ring_Za, const uint16_t *ring_Cb,
    const uint16_t *ring_Zb, const uint16_t *Ba, const uint16_t *Bb,
    const uint16_t *rms_w, void *kv_comp, int64_t n_cap,
    const uint8_t *kI, const uint8_t *qI, const uint16_t *wI,
    const uint16_t *q, const uint16_t *swa_ring, const float *sink,
    int32_t *idx_out, uint16_t *out, float *lse, void *workspace,
    size_t workspace_bytes, void *stream);

/*
 * csa_layer_decode_append — csa_layer_decode whose first kernel also stores
 * the step's new rows into the caches it then reads (a serving loop's
 * per-step cache append, without launches of its own):
 *
 *   swa_new [B][512] bf16: the window row of position t = q_pos[b], stored
 *           into swa_ring slot t mod W before the attention reads the ring;
 *   kI_new  [B][128] e4m3, or NULL: where (t+1) % m == 0, the indexer key of
 *           the entry completing at t, i = (t+1)/m - 1, stored into kI[b, i]
 *           before the indexer reads it (other rows of kI_new are not read;
 *           an i >= n_cap is not stored and is reported by step 1 as for
 *           csa_layer_decode).
 *
 * Sequences with q_pos[b] < 0 store nothing.  swa_ring and kI are written,
 * hence not const here; every other argument and the result are as for
 * csa_layer_decode.  Errors: CSA_ERR_INVALID_ARG for a NULL or unaligned
 * swa_new or an unaligned kI_new; CSA_ERR_UNSUPPORTED for kI_new with
 * index_format 1 (FP4 index keys live in planes, see above).
 */
csa_status csa_layer_decode_append(
    const csa_params *p, int32_t B, const int32_t *q_pos,
    const uint16_t *swa_new, const uint8_t *kI_new,
    const uint16_t *ring_Ca, const uint16_t *ring_Za, const uint16_t *ring_Cb,
    const uint16_t *ring_Zb, const uint16_t *Ba, const uint16_t *Bb,
    const uint16_t *rms_w, void *kv_comp, int64_t n_cap,
    uint8_t *kI, const uint8_t *qI, const uint16_t *wI,
    const uint16_t *q, uint16_t *swa_ring, const float *sink,
    int32_t *idx_out, uint16_t *out, float *lse, void *workspace,
    size_t workspace_bytes, void *stream);

/*
 * csa_index_key_src — the inputs of the lightning indexer's own key
 * compressor (width 128; the steps of csa_compress_indexer_keys), for the
 * layer calls that compute their indexer keys themselves.  [hca_csa]
 * "CSA：轻压缩 + 稀疏选择": the indexer compresses its keys at its own width
 * with the main cache's entry numbering, then rotates them by H_128/sqrt(128)
 * and stores FP8 codes.
 *
 * Decode (csa_layer_decode_with_keys): CIa, ZIa, CIb, ZIb are staging rings
 *   [B][2m][128] bf16 laid out as the main compressor's ring (the row of
 *   token u in slot u mod 2m, holding tokens t-2m+1..t); CIb_prev and
 *   ZIb_prev are not read.
 * Prefill (csa_layer_prefill_with_keys): CIa, ZIa, CIb, ZIb are [B][Q][128]
 *   bf16 rows of the chunk's tokens; CIb_prev, ZIb_prev [B][m][128] the rows
 *   of the block before the chunk, NULL iff pos0 == 0.
 * BIa, BIb [m][128] bf16 slot biases; rms_wI [128] bf16 RMSNorm weight.
 * All pointers are device pointers owned by the caller, 16-byte aligned.
 */
typedef struct csa_index_key_src {
  const uint16_t *CIa, *ZIa, *CIb, *ZIb;
  const uint16_t *CIb_prev, *ZIb_prev;
  const uint16_t *BIa, *BIb;
  const uint16_t *rms_wI;
} csa_index_key_src;

/*
 * csa_layer_decode_with_keys — csa_layer_decode_append whose indexer key is
 * computed by the call instead of given: one decode step that needs nothing
 * but the staging rings, the caches and the queries.  The step's first
 * kernel (the one that clears the counters) stores swa_new (if not NULL)
 * into swa_ring slot t mod W and, where (t+1) % m == 0, computes the key of
 * entry i = (t+1)/m - 1 from the key compressor's ring (*keys) into kI[b, i]
 * before the indexer reads it; then the steps of csa_layer_decode.  keys is
 * a host pointer to the struct (read during the call); its arrays and every
 * other pointer are as for csa_layer_decode_append, except that swa_new may
 * be NULL.  Errors: those of csa_layer_decode; CSA_ERR_INVALID_ARG for a
 * NULL keys or a NULL or unaligned array in it; CSA_ERR_UNSUPPORTED for
 * index_format 1 (this compressor writes E4M3 keys).
 */
csa_status csa_layer_decode_with_keys(
    const csa_params *p, int32_t B, const int32_t *q_pos,
    const uint16_t *swa_new, const csa_index_key_src *keys,
    const uint16_t *ring_Ca, const uint16_t *ring_Za, const uint16_t *ring_Cb,
    const uint16_t *ring_Zb, const uint16_t *Ba, const uint16_t *Bb,
    const uint16_t *rms_w, void *kv_comp, int64_t n_cap,
    uint8_t *kI, const uint8_t *qI, const uint16_t *wI,
    const uint16_t *q, uint16_t *swa_ring, const float *sink,
    int32_t *idx_out, uint16_t *out, float *lse, void *workspace,
    size_t workspace_bytes, void *stream);

/*
 * csa_layer_prefill — one chunk of Q query tokens at positions pos0..pos0+Q-1
 * (pos0 a multiple of m, given on the host), causal per query.
 * [hca_csa] "在 SGLang 里的落点" (large-batch prefill has the decode
 * semantics); future entries masked before top-k [KV 压缩] §9.8.
 *
 *   1. compress the chunk: entries pos0/m .. (pos0+Q)/m - 1 (a trailing
 *      incomplete block produces no entry) → kv_comp, as csa_compress;
 *   2. index + top-k for each query t over its own V(t);
 *   3. sparse attention with the linear window.
 *
 * Ca/Za/Cb/Zb : [B][Q][512] bf16 rows of the chunk's tokens.
 * Cb_prev/Zb_prev: [B][m][512] rows of the block before the chunk, NULL iff
 *         pos0 == 0.
 * kI    : must already hold entries 0..(pos0+Q)/m - 1.
 * qI [B][Q][64][128], wI [B][Q][64], q [B][Q][64][512].
 * swa   : [B][W-1+Q][512] bf16, row j = position pos0-(W-1)+j (rows before
 *         position 0 are never read).
 * idx_out [B][Q][topk], out [B][Q][64][512], lse [B][Q][64] or NULL.
 */
csa_status csa_layer_prefill(
    const csa_params *p, int32_t B, int32_t Q, int64_t pos0,
    const uint16_t *Ca, const uint16_t *Za, const uint16_t *Cb,
    const uint16_t *Zb, const uint16_t *Cb_prev, const uint16_t *Zb_prev,
    const uint16_t *Ba, const uint16_t *Bb, const uint16_t *rms_w,
    void *kv_comp, int64_t n_cap, const uint8_t *kI, const uint8_t *qI,
    const uint16_t *wI, const uint16_t *q, const uint16_t *swa,
    const float *sink, int32_t *idx_out, uint16_t *out, float *lse,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * csa_layer_prefill_with_keys — csa_layer_prefill that also computes the
 * chunk's indexer keys: the compressor launch of step 1 writes, beside each
 * entry i = pos0/m .. (pos0+Q)/m - 1 of kv_comp, its indexer key into
 * kI[b, i] from *keys (prefill layout, see csa_index_key_src), so that kI
 * need only hold entries 0..pos0/m - 1 beforehand.  keys is a host pointer
 * read during the call; kI is written, hence not const.  Errors: those of
 * csa_layer_prefill; CSA_ERR_INVALID_ARG for a NULL keys, a NULL or
 * unaligned array in it, or CIb_prev/ZIb_prev not NULL exactly when
 * pos0 == 0; CSA_ERR_UNSUPPORTED for index_format 1.
 */
csa_status csa_layer_prefill_with_keys(
    const csa_params *p, int32_t B, int32_t Q, int64_t pos0,
    const uint16_t *Ca, const uint16_t *Za, const uint16_t *Cb,
    const uint16_t *Zb, const uint16_t *Cb_prev, const uint16_t *Zb_prev,
    const uint16_t *Ba, const uint16_t *Bb, const uint16_t *rms_w,
    const csa_index_key_src *keys, void *kv_comp, int64_t n_cap, uint8_t *kI,
    const uint8_t *qI, const uint16_t *wI, const uint16_t *q,
    const uint16_t *swa, const float *sink, int32_t *idx_out, uint16_t *out,
    float *lse, void *workspace, size_t workspace_bytes, void *stream);

/*
 * csa_hca_layer_decode — one decode step of an HCA layer (block size p->m,
 * 128 in the pages; no indexer) for B sequences ([hca_csa] "HCA：同一个算子，
 * 关掉重叠"; [CSA2 详解] §9: the layer reads every causally visible entry):
 *   1. csa_compress_single_step with the step's token rows C, Z: the token
 *      joins its block's online state, and a token that completes block i
 *      writes entry i to kv_comp;
 *   2. csa_sparse_attn with idx = NULL over the ring window swa_ring and the
 *      entries 0 .. floor((t+1)/m)-1, the one just written included.
 * Arguments are those of the two calls (kv_comp: [B][n_cap][512] bf16,
 * kv_stride_b = n_cap*512).  Workspace: csa_workspace_size(
 * CSA_OP_HCA_LAYER_DECODE, p, B, 1, n_cap) bytes or NULL (see
 * csa_sparse_attn).  Stage events (csa_set_trace_events): 1 after the
 * compressor, 4 after the attention (2 and 3 with 1).
 */
csa_status csa_hca_layer_decode(const csa_params *p, int32_t B,
                                const int32_t *q_pos, const uint16_t *C,
                                const uint16_t *Z, const uint16_t *bias,
                                const uint16_t *rms_w, float *state,
                                uint16_t *kv_comp, int64_t n_cap,
                                const uint16_t *q, const uint16_t *swa_ring,
                                const float *sink, uint16_t *out, float *lse,
                                void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * Optional stage tracing, for profiling.  With events != NULL (n_events == 5
 * cudaEvent_t handles passed as void*), every csa_layer_decode(_append,
 * _with_keys) and csa_layer_prefill(_with_keys) call records events[0] on
 * its stream before its first kernel and events[s] after stage s: 1 the
 * first kernel (counters cleared, new rows stored, indexer key computed) and
 * the compressor, 2 indexer scores, 3 top-k, 4 sparse attention.
 * csa_index_topk, csa_index_topk_static, csa_index_topk_pool and
 * csa_reindex_topk record events[1] before their indexer kernel (after
 * clearing their workspace), events[2] after it and events[3] after their
 * top-k launches.  events == NULL turns tracing off.  The setting is
 * process-wide; set it only while no traced call runs on another thread.
 */
csa_status csa_set_trace_events(void *const *events, int32_t n_events);

/* Number of kernels this library has launched in this process so far. */
uint64_t csa_launch_count(void);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device (CSA_OK, CSA_ERR_TIMEOUT or CSA_ERR_INDEX_RANGE), or
 * CSA_ERR_CUDA if the stream reported an error.
 */
csa_status csa_check_status(void *stream);

/*
 * csa_test_set_wait_fault — test-only switch for the failure path of the
 * bounded device waits (failure detection: every wait of the library's
 * kernels gives up after a limit, records CSA_ERR_TIMEOUT and lets its kernel
 * finish; a CTA still releases its tensor memory and waits for its own copies
 * in flight).  Off by default; nothing but this call turns it on.
 *
 * wait_limit_us: the limit of every device wait on the current device, in
 *   microseconds; 0 restores the default (2 s).
 * faults: OR of the CSA_TEST_FAULT_* bits, each withholding one signal in
 *   the kernels of later calls so that a wait must give up:
 *     INDEXER  the lightning indexer's producer never loads its first key
 *              tile (csa_index_topk and the layer and pool calls);
 *     TOPK     a top-k cluster's rank 0 never sends its first crossing (rows
 *              of more than 4096 keys);
 *     ATTN     the sparse attention's MMA thread never announces the first
 *              tile's scores (every form: single CTA, cluster, split-KV).
 *   A non-zero faults needs a non-zero wait_limit_us.
 * Synchronises the device first.  Process-wide per device: set it only while
 * no other call runs.  Errors: CSA_ERR_INVALID_ARG for unknown bits or faults
 * without a limit; CSA_ERR_CUDA.
 */
#define CSA_TEST_FAULT_INDEXER 1u
#define CSA_TEST_FAULT_TOPK 2u
#define CSA_TEST_FAULT_ATTN 4u
csa_status csa_test_set_wait_fault(uint32_t wait_limit_us, uint32_t faults);

/* Static, human-readable name of a status code. */
const char *csa_status_string(csa_status s);

#ifdef __cplusplus
}
#endif

#endif /* LIBCSA_CSA_H */
