/*
 * CSA oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded fp64 CPU statement of what one CSA layer's
 * hot path computes.  It exists to check the CUDA library against; only the
 * tests, the package's smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * Inputs are taken as their raw storage bits (bf16 as uint16, FP8 E4M3 as
 * uint8, sink as fp32) and decoded here from the format definitions; all
 * arithmetic is then in double, in the order the pages state it.
 *
 * Pages cited (by title):
 *   [hca_csa]   "CSA / HCA" (zdszero.github.io, hca_csa)
 *   [KV 压缩]   "DeepSeek-V4 的 KV 压缩：从删 token 误解到预算检索"
 *   [CSA2 详解] "DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2：从模型原理到推理基础设施"
 *   [结构对比]  "DeepSeek 注意力结构对比：MHA、GQA、MLA、DSA、CSA、HCA、CSA2"
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- storage formats ---------------------------------------------------- */

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
double orc_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* FP8 E4M3 ("fn": no infinities, S.1111.111 is NaN): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal. */
double orc_e4m3(uint8_t bits) {
  int sign = bits >> 7;
  int e = (bits >> 3) & 0xF;
  int f = bits & 0x7;
  double mag;
  if (e == 0xF && f == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)f / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)f / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* ---- compressor ([hca_csa] "CSA 的重叠窗口") ------------------------------ */

/*
 * Soft pooling of entry i, before Norm and RoPE.  For each channel d the 2m
 * logits are Za[r][d] + Ba[r][d] (block i) and Zb[r][d] + Bb[r][d] (block
 * i-1); Softmax_row normalises over all 2m of them, and the weighted C rows
 * are summed.  With has_prev == 0 (entry 0) the block-(i-1) logits are -inf
 * and their C rows are 0, as the page states for i = 0.
 *   Ca, Za : [m][D] rows of block i;  Cb, Zb : [m][D] rows of block i-1.
 *   Ba, Bb : [m][D].                  x     : [D] output.
 */
void orc_compress_pool(int m, int D, int has_prev, const uint16_t *Ca,
                       const uint16_t *Za, const uint16_t *Cb,
                       const uint16_t *Zb, const uint16_t *Ba,
                       const uint16_t *Bb, double *x) {
  double logit[64], value[64];
  for (int d = 0; d < D; ++d) {
    int n = 0;
    for (int r = 0; r < m; ++r) {
      logit[n] = orc_bf16(Za[r * D + d]) + orc_bf16(Ba[r * D + d]);
      value[n] = orc_bf16(Ca[r * D + d]);
      ++n;
    }
    for (int r = 0; r < m; ++r) {
      if (has_prev) {
        logit[n] = orc_bf16(Zb[r * D + d]) + orc_bf16(Bb[r * D + d]);
        value[n] = orc_bf16(Cb[r * D + d]);
      } else {
        logit[n] = -INFINITY;
        value[n] = 0.0;
      }
      ++n;
    }
    double mx = -INFINITY;
    for (int j = 0; j < n; ++j)
      if (logit[j] > mx) mx = logit[j];
    double num = 0.0, den = 0.0;
    for (int j = 0; j < n; ++j) {
      double e = exp(logit[j] - mx);
      num += e * value[j];
      den += e;
    }
    x[d] = num / den;
  }
}

/* RMSNorm ("Norm" in the C_i^Comp equation): y = x / sqrt(mean(x^2) + eps) * w. */
void orc_rmsnorm(int D, const double *x, const uint16_t *w, double eps,
                 double *y) {
  double ss = 0.0;
  for (int d = 0; d < D; ++d) ss += x[d] * x[d];
  double inv = 1.0 / sqrt(ss / (double)D + eps);
  for (int d = 0; d < D; ++d) y[d] = x[d] * inv * orc_bf16(w[d]);
}

/* Partial RoPE on the last R channels, interleaved pairs (D-R+2j, D-R+2j+1),
 * rotated by angle pos * theta^(-2j/R) (in place). */
void orc_rope(int D, int R, double theta, double pos, double *y) {
  for (int j = 0; j < R / 2; ++j) {
    double freq = pow(theta, -2.0 * (double)j / (double)R);
    double phi = pos * freq;
    double c = cos(phi), s = sin(phi);
    int a = D - R + 2 * j;
    double u = y[a], v = y[a + 1];
    y[a] = u * c - v * s;
    y[a + 1] = u * s + v * c;
  }
}

/* One compressed entry i: RoPE(Norm(pool)), RoPE position m*i (the first
 * token of the entry's own block, [CSA2 详解] §7.4). */
void orc_compress_entry(int m, int D, int R, double theta, double eps,
                        int64_t i, const uint16_t *Ca, const uint16_t *Za,
                        const uint16_t *Cb, const uint16_t *Zb,
                        const uint16_t *Ba, const uint16_t *Bb,
                        const uint16_t *w, double *out) {
  double *x = (double *)malloc(sizeof(double) * (size_t)D);
  orc_compress_pool(m, D, i > 0, Ca, Za, Cb, Zb, Ba, Bb, x);
  orc_rmsnorm(D, x, w, eps, out);
  orc_rope(D, R, theta, (double)m * (double)i, out);
  free(x);
}

/* ---- non-overlapped compressor ([hca_csa] "HCA：同一个算子，关掉重叠";
 * [CSA2 详解] §7.2 and §7.5) ----------------------------------------------- */

/*
 * Entry i from the m rows of its own block only: for each channel d the m
 * logits are Z[r][d] + B[r][d] (HCA; B == NULL: no position bias, as in
 * CSA2), Softmax_row normalises over them and weights the C rows; then
 * RMSNorm and RoPE at position m*i as for the overlapped compressor.  With
 * m = 1 the one softmax weight is 1 and the entry is RoPE(Norm(C)).
 *   C, Z : [m][D] rows of block i;  B : [m][D] or NULL;  out : [D].
 */
void orc_compress_single_entry(int m, int D, int R, double theta, double eps,
                               int64_t i, const uint16_t *C, const uint16_t *Z,
                               const uint16_t *B, const uint16_t *w,
                               double *out) {
  double *x = (double *)malloc(sizeof(double) * (size_t)D);
  double *logit = (double *)malloc(sizeof(double) * (size_t)m);
  for (int d = 0; d < D; ++d) {
    double mx = -INFINITY;
    for (int r = 0; r < m; ++r) {
      logit[r] = orc_bf16(Z[r * D + d]) + (B ? orc_bf16(B[r * D + d]) : 0.0);
      if (logit[r] > mx) mx = logit[r];
    }
    double num = 0.0, den = 0.0;
    for (int r = 0; r < m; ++r) {
      double e = exp(logit[r] - mx);
      num += e * orc_bf16(C[r * D + d]);
      den += e;
    }
    x[d] = num / den;
  }
  orc_rmsnorm(D, x, w, eps, out);
  orc_rope(D, R, theta, (double)m * (double)i, out);
  free(logit);
  free(x);
}

/* ---- indexer keys ([hca_csa] "CSA：轻压缩 + 稀疏选择": the indexer has a
 * compressor of its own at head_dim 128, followed by a Hadamard rotation so
 * that the keys quantise well to FP8) ------------------------------------- */

/* y = H_n x / sqrt(n): H_n is the Sylvester Hadamard matrix (n a power of
 * two), H_1 = [1], H_2k = [[H_k, H_k], [H_k, -H_k]], whose entry (r, c) is
 * (-1)^(number of bits set in r AND c).  Dense product, as the definition. */
void orc_hadamard(int n, const double *x, double *y) {
  for (int r = 0; r < n; ++r) {
    double acc = 0.0;
    for (int c = 0; c < n; ++c) {
      unsigned v = (unsigned)(r & c);
      int parity = 0;
      while (v) {
        parity ^= (int)(v & 1u);
        v >>= 1;
      }
      acc += parity ? -x[c] : x[c];
    }
    y[r] = acc / sqrt((double)n);
  }
}

/* The E4M3 code nearest to x: ties go to the code with an even mantissa (the
 * last bit clear), magnitudes past the largest finite value (448) give +-448,
 * NaN gives 0x7F.  Found by comparing with every finite code's value. */
uint8_t orc_to_e4m3(double x) {
  if (x != x) return 0x7F;
  const uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0x00;
  const double a = fabs(x);
  int best = 0;
  double best_err = a;  /* code 0 is +0 */
  for (int c = 1; c <= 0x7E; ++c) {
    const double err = fabs(orc_e4m3((uint8_t)c) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/* One indexer key entry i: the compressor's steps at width Dk (pool, RMSNorm
 * with the key compressor's weight, RoPE on the last R channels at position
 * m*i), then the Hadamard rotation, then E4M3.  pre receives the rotated
 * values before rounding, codes the stored bytes. */
void orc_index_key_entry(int m, int Dk, int R, double theta, double eps,
                         int64_t i, const uint16_t *Ca, const uint16_t *Za,
                         const uint16_t *Cb, const uint16_t *Zb,
                         const uint16_t *Ba, const uint16_t *Bb,
                         const uint16_t *w, double *pre, uint8_t *codes) {
  double *x = (double *)malloc(sizeof(double) * (size_t)Dk);
  double *y = (double *)malloc(sizeof(double) * (size_t)Dk);
  orc_compress_pool(m, Dk, i > 0, Ca, Za, Cb, Zb, Ba, Bb, x);
  orc_rmsnorm(Dk, x, w, eps, y);
  orc_rope(Dk, R, theta, (double)m * (double)i, y);
  orc_hadamard(Dk, y, pre);
  for (int d = 0; d < Dk; ++d) codes[d] = orc_to_e4m3(pre[d]);
  free(x);
  free(y);
}

/* ---- FP4 cache entries ([CSA2 详解] §16.1: a Main KV entry is 512 FP4
 * values with one 1-byte E4M3 scale per 16 values, 288 bytes) ------------- */

/* Value of an E2M1 code: bit 3 the sign, bits 2..1 the exponent (bias 1),
 * bit 0 the mantissa; exponent 0 is subnormal.  Magnitudes 0, 0.5, 1, 1.5,
 * 2, 3, 4, 6. */
double orc_e2m1(uint8_t code) {
  const int e = (code >> 1) & 3, m = code & 1;
  const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return (code & 8) ? -mag : mag;
}

/* The E2M1 code nearest to x: ties go to the code with an even mantissa,
 * magnitudes past 6 give +-6, the sign is kept (a small negative x gives
 * -0).  Found by comparing with every code's value. */
uint8_t orc_to_e2m1(double x) {
  const uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 8 : 0;
  const double a = fabs(x);
  int best = 0;
  double best_err = a;
  for (int c = 1; c <= 7; ++c) {
    const double err = fabs(orc_e2m1((uint8_t)c) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/*
 * One Main KV entry of D bf16 values in the FP4 layout.  Bytes 0 .. D/2-1:
 * the E2M1 codes, channel 2j in the low nibble of byte j and channel 2j+1 in
 * the high nibble; bytes D/2 .. D/2 + D/16 - 1: the E4M3 scales, scale g for
 * channels 16g .. 16g+15.  Scale of a group: the E4M3 code nearest to
 * amax / 6 (amax the group's largest magnitude), the quotient formed in
 * binary32, as the kernel forms it, because it decides a code; code of a
 * channel: E2M1 of x / s, the quotient again in binary32; a group whose
 * scale is zero gets zero codes.  The stored value is s * e2m1(code).
 */
void orc_quantize_kv_fp4(int D, const uint16_t *x, uint8_t *out) {
  for (int g = 0; g < D / 16; ++g) {
    float amax = 0.0f;
    for (int c = 16 * g; c < 16 * g + 16; ++c) {
      const float v = (float)fabs(orc_bf16(x[c]));
      if (v > amax) amax = v;
    }
    const float q = amax / 6.0f;
    const uint8_t sc = orc_to_e4m3((double)q);
    out[D / 2 + g] = sc;
    const float s = (float)orc_e4m3(sc);
    for (int c = 16 * g; c < 16 * g + 16; c += 2) {
      uint8_t lo = 0, hi = 0;
      if (s != 0.0f) {
        lo = orc_to_e2m1((double)((float)orc_bf16(x[c]) / s));
        hi = orc_to_e2m1((double)((float)orc_bf16(x[c + 1]) / s));
      }
      out[c / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

/* The D values an FP4 entry stands for: s * e2m1(code). */
void orc_dequantize_kv_fp4(int D, const uint8_t *in, double *x) {
  for (int c = 0; c < D; ++c) {
    const uint8_t code = (uint8_t)((in[c / 2] >> (4 * (c & 1))) & 0xF);
    x[c] = orc_e4m3(in[D / 2 + c / 16]) * orc_e2m1(code);
  }
}

/* ---- FP4 indexer keys and queries ([CSA2 详解] §16.2) --------------------
 * The CSA2 indexer holds its keys (and forms its queries) as 128 FP4 E2M1
 * values with one 1-byte E8M0 scale per 32 values (68 bytes a key).  The
 * pages do not say how the power-of-two scale is rounded; the reading here:
 * the smallest power of two s with 6 * s >= amax (6 is E2M1's largest value),
 * so every x / s lies within E2M1's range and no code saturates. */

/* E8M0 byte of a block whose largest magnitude is amax: e + 127 for the
 * smallest e in -127..127 with 6 * 2^e >= amax (a zero block: byte 0). */
uint8_t orc_e8m0_scale(double amax) {
  int e = -127;
  while (e < 127 && 6.0 * ldexp(1.0, e) < amax) ++e;
  return (uint8_t)(e + 127);
}

/* Value of an E8M0 byte (255, the format's NaN, is never produced here). */
double orc_e8m0(uint8_t b) { return ldexp(1.0, (int)b - 127); }

/* One row of D bf16 values: codes[j] holds channel 2j in its low nibble and
 * 2j+1 in its high nibble; scales[g] is the E8M0 byte of channels
 * 32g .. 32g+31; a channel's code is the E2M1 code nearest to x / s (ties to
 * the even code, sign kept; the quotient is exact, s being a power of two). */
void orc_quantize_index_fp4(int D, const uint16_t *x, uint8_t *codes, uint8_t *scales) {
  for (int g = 0; g < D / 32; ++g) {
    double amax = 0.0;
    for (int c = 32 * g; c < 32 * g + 32; ++c)
      if (fabs(orc_bf16(x[c])) > amax) amax = fabs(orc_bf16(x[c]));
    scales[g] = orc_e8m0_scale(amax);
    const double s = orc_e8m0(scales[g]);
    for (int c = 32 * g; c < 32 * g + 32; c += 2) {
      const uint8_t lo = orc_to_e2m1(orc_bf16(x[c]) / s);
      const uint8_t hi = orc_to_e2m1(orc_bf16(x[c + 1]) / s);
      codes[c / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

/* n such rows, row r at x + r*D, codes + r*D/2, scales + r*D/32. */
void orc_quantize_index_fp4_rows(int64_t n, int D, const uint16_t *x, uint8_t *codes, uint8_t *scales) {
  for (int64_t r = 0; r < n; ++r)
    orc_quantize_index_fp4(D, x + r * D, codes + r * (D / 2), scales + r * (D / 32));
}

/* The D values such a row stands for: e8m0(scale of the block) * e2m1(code). */
void orc_dequantize_index_fp4(int D, const uint8_t *codes, const uint8_t *scales, double *x) {
  for (int c = 0; c < D; ++c)
    x[c] = orc_e8m0(scales[c / 32]) * orc_e2m1((uint8_t)((codes[c / 2] >> (4 * (c & 1))) & 0xF));
}

/* n such rows decoded, row r at x + r*D. */
void orc_dequantize_index_fp4_rows(int64_t n, int D, const uint8_t *codes, const uint8_t *scales, double *x) {
  for (int64_t r = 0; r < n; ++r)
    orc_dequantize_index_fp4(D, codes + r * (D / 2), scales + r * (D / 32), x + r * D);
}

/* ---- visibility ([KV 压缩] §9.8) ---------------------------------------- */

/* Entry s covers tokens up to m*s + m - 1, so the query at position t sees
 * entries s with (s+1)*m <= t+1: the count is floor((t+1)/m). */
int64_t orc_visible(int64_t t, int m) { return (t + 1) / m; }

/* ---- lightning indexer ([hca_csa] equation I_{t,s}) ---------------------- */

/* scores[s] = sum_h w[h] * ReLU(q[h,:] . k[s,:]) for s < V.
 *   q : [H][Dk] e4m3;  w : [H] bf16;  k : [V][Dk] e4m3. */
void orc_index_scores(int H, int Dk, int64_t V, const uint8_t *q,
                      const uint16_t *w, const uint8_t *k, double *scores) {
  double *qd = (double *)malloc(sizeof(double) * (size_t)H * (size_t)Dk);
  double *kd = (double *)malloc(sizeof(double) * (size_t)Dk);
  for (int i = 0; i < H * Dk; ++i) qd[i] = orc_e4m3(q[i]);
  for (int64_t s = 0; s < V; ++s) {
    for (int c = 0; c < Dk; ++c) kd[c] = orc_e4m3(k[s * Dk + c]);
    double total = 0.0;
    for (int h = 0; h < H; ++h) {
      double dot = 0.0;
      for (int c = 0; c < Dk; ++c) dot += qd[h * Dk + c] * kd[c];
      double relu = dot > 0.0 ? dot : 0.0;
      total += orc_bf16(w[h]) * relu;
    }
    scores[s] = total;
  }
  free(kd);
  free(qd);
}

/* The same score over values already decoded to doubles (the FP4 indexer):
 *   q : [H][Dk];  w : [H] bf16;  k : [V][Dk]. */
void orc_index_scores_f64(int H, int Dk, int64_t V, const double *q, const uint16_t *w, const double *k,
                          double *scores) {
  for (int64_t s = 0; s < V; ++s) {
    double total = 0.0;
    for (int h = 0; h < H; ++h) {
      double dot = 0.0;
      for (int c = 0; c < Dk; ++c) dot += q[h * Dk + c] * k[s * Dk + c];
      total += orc_bf16(w[h]) * (dot > 0.0 ? dot : 0.0);
    }
    scores[s] = total;
  }
}

/* ---- top-k ---------------------------------------------------------------- */

typedef struct {
  double score;
  int64_t index;
} orc_scored;

/* Larger score first; equal scores: smaller entry index first. */
static int orc_by_score(const void *pa, const void *pb) {
  const orc_scored *a = (const orc_scored *)pa, *b = (const orc_scored *)pb;
  if (a->score > b->score) return -1;
  if (a->score < b->score) return 1;
  return (a->index < b->index) ? -1 : (a->index > b->index);
}

static int orc_by_index(const void *pa, const void *pb) {
  int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
  return (a > b) - (a < b);
}

/* The min(k, V) entries with the largest scores (ties toward the smaller
 * index), written in ascending entry order, then -1 up to k slots.  Returns
 * the number of selected entries.  The ascending (position) order follows [结构对比]'s CSA2 section. */
int orc_topk(int64_t V, int k, const double *scores, int32_t *idx) {
  orc_scored *all = (orc_scored *)malloc(sizeof(orc_scored) * (size_t)(V > 0 ? V : 1));
  for (int64_t s = 0; s < V; ++s) {
    all[s].score = scores[s];
    all[s].index = s;
  }
  qsort(all, (size_t)V, sizeof(orc_scored), orc_by_score);
  int n = (int)(V < k ? V : k);
  for (int j = 0; j < n; ++j) idx[j] = (int32_t)all[j].index;
  qsort(idx, (size_t)n, sizeof(int32_t), orc_by_index);
  for (int j = n; j < k; ++j) idx[j] = -1;
  free(all);
  return n;
}

/* ---- joint softmax with sink ([hca_csa] o_{t,i} equation) ---------------- */

/*
 * One query: H heads of width D attend to n_rows shared K=V rows.
 *   l_{h,j} = sm_scale * q[h,:] . row_j
 *   out[h,:] = sum_j e^{l_hj - M} row_j / (sum_j e^{l_hj - M} + e^{sink_h - M})
 * with M = max(max_j l_hj, sink_h); lse[h] = M + log(denominator).  The sink
 * is one more logit in the shared denominator with a zero value row.
 *   q : [H][D] bf16;  rows : [n_rows][D] bf16 (already gathered);  sink : [H].
 *   out : [H][D];  lse : [H] (may be NULL).
 */
void orc_attend(int H, int D, int n_rows, const uint16_t *q,
                const uint16_t *rows, const float *sink, double sm_scale,
                double *out, double *lse) {
  size_t n = (size_t)(n_rows > 0 ? n_rows : 1);
  double *logit = (double *)malloc(sizeof(double) * n);
  double *weight = (double *)malloc(sizeof(double) * n);
  for (int h = 0; h < H; ++h) {
    double mx = (double)sink[h];
    for (int j = 0; j < n_rows; ++j) {
      double dot = 0.0;
      for (int c = 0; c < D; ++c)
        dot += orc_bf16(q[h * D + c]) * orc_bf16(rows[(size_t)j * D + c]);
      logit[j] = sm_scale * dot;
      if (logit[j] > mx) mx = logit[j];
    }
    double den = exp((double)sink[h] - mx);
    for (int j = 0; j < n_rows; ++j) {
      weight[j] = exp(logit[j] - mx);
      den += weight[j];
    }
    for (int c = 0; c < D; ++c) {
      double num = 0.0;
      for (int j = 0; j < n_rows; ++j)
        num += weight[j] * orc_bf16(rows[(size_t)j * D + c]);
      out[h * D + c] = num / den;
    }
    if (lse) lse[h] = mx + log(den);
  }
  free(weight);
  free(logit);
}

/* ---- array helpers for the Python wrapper -------------------------------- */

void orc_decode_bf16(int64_t n, const uint16_t *in, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16(in[i]);
}

void orc_decode_e4m3(int64_t n, const uint8_t *in, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3(in[i]);
}
