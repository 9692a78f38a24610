// The non-overlapped compressor of HCA and CSA2 layers.  Page "CSA / HCA"
// (zdszero, hca_csa), section "HCA：同一个算子，关掉重叠" (one stream C, Z, B;
// Softmax_row over the m slots of the entry's own block, then Norm and
// RoPE); "DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §7.2 (CSA2: the same
// pooling without the slot bias) and §7.5 (ratio 1: the softmax weight is 1);
// RoPE at the first token of the block (§7.4).  The decode form keeps, per
// sequence and channel, a running (max, sum, weighted sum) over the block's
// tokens so far, the online-softmax state of the HCA compressor described in
// "CSA / HCA", section "KV cache：成品与原料", instead of a ring of raw rows.
//
// Bulk: one 256-thread CTA per (entry, sequence).  The rows of C and Z stream
// through shared memory in stages of up to 8 rows (one bulk copy of each, a
// ring of 4 stages in flight; the slot biases of the next stage are loaded
// while one is computed); four groups of 64 threads take every fourth row of
// a stage with an online softmax in fp32; group 0 merges the partial states
// and finishes the entry (RMSNorm, RoPE, bf16 store).  (Two CTAs per entry,
// each with half of the rows and a merge through distributed shared memory,
// were measured slower at HCA's m = 128: 69 against 54 us for 1024 entries.)
// Step: one 64-thread CTA per sequence updates its state with the step's
// token and, when the token closes a block, finishes the entry.  The
// exponentials and the final divide are the hardware approximations (a few
// ulp, far inside the bf16 output's rounding).
#include "compress.cuh"

namespace csa {
namespace {

constexpr int kGroupThreads = kDim / 8;  // 64: 8 channels per thread
constexpr int kRowGroups = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kStageRows = 8;  // rows of C (and of Z) per stage
#ifndef CSA_HCA_STAGES
#define CSA_HCA_STAGES 4
#endif
#ifndef CSA_HCA_CTAS_PER_SM
#define CSA_HCA_CTAS_PER_SM 3
#endif
constexpr int kStages = CSA_HCA_STAGES;  // stages in flight
constexpr uint32_t kStageBytes = kStageRows * kDim * 2;
constexpr size_t kBulkSmem = 2 * kStages * kStageBytes + kStages * sizeof(uint64_t);  // C and Z rings, barriers
static_assert((kRowGroups - 1) * 3 * kDim * sizeof(float) <= kStages * kStageBytes, "merge states fit the C ring");

// Folds one row's logits and values into the running state of 8 channels.
__device__ __forceinline__ void online_add(const float (&logit)[8], const float (&c)[8], float (&mx)[8],
                                           float (&den)[8], float (&num)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float nm = fmaxf(mx[j], logit[j]);
    const float sc = ex2_approx((mx[j] - nm) * kLog2e);  // 0 while the state is empty (mx = -inf)
    const float p = ex2_approx((logit[j] - nm) * kLog2e);
    num[j] = fmaf(num[j], sc, p * c[j]);
    den[j] = fmaf(den[j], sc, p);
    mx[j] = nm;
  }
}

// Folds two rows' logits and values into the running state of 8 channels:
// one rescale of the state per pair (the larger of the two rows' logits and
// the running maximum), and each exponent's argument as one fused
// multiply-add of the logit with log2(e) against the new maximum's product;
// the multiply-adds run on channel pairs (packed fp32, each component
// rounded as the scalar operation rounds it).
__device__ __forceinline__ void online_add2(const float (&l0)[8], const float (&c0)[8], const float (&l1)[8],
                                            const float (&c1)[8], float (&mx)[8], float (&den)[8], float (&num)[8]) {
  const float2 k2 = make_float2(kLog2e, kLog2e), nk2 = make_float2(-kLog2e, -kLog2e);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float nm0 = fmaxf(mx[j], fmaxf(l0[j], l1[j])), nm1 = fmaxf(mx[j + 1], fmaxf(l0[j + 1], l1[j + 1]));
    const float2 nk = __fmul2_rn(make_float2(nm0, nm1), nk2);  // -max * log2(e)
    const float2 as = __ffma2_rn(make_float2(mx[j], mx[j + 1]), k2, nk);  // -inf while the state is empty
    const float2 a0 = __ffma2_rn(make_float2(l0[j], l0[j + 1]), k2, nk);
    const float2 a1 = __ffma2_rn(make_float2(l1[j], l1[j + 1]), k2, nk);
    const float2 sc = make_float2(ex2_approx(as.x), ex2_approx(as.y));
    const float2 p0 = make_float2(ex2_approx(a0.x), ex2_approx(a0.y));
    const float2 p1 = make_float2(ex2_approx(a1.x), ex2_approx(a1.y));
    const float2 t = __ffma2_rn(p0, make_float2(c0[j], c0[j + 1]), __fmul2_rn(p1, make_float2(c1[j], c1[j + 1])));
    const float2 nu = __ffma2_rn(make_float2(num[j], num[j + 1]), sc, t);
    const float2 de = __ffma2_rn(make_float2(den[j], den[j + 1]), sc, __fadd2_rn(p0, p1));
    num[j] = nu.x;
    num[j + 1] = nu.y;
    den[j] = de.x;
    den[j + 1] = de.y;
    mx[j] = nm0;
    mx[j + 1] = nm1;
  }
}

// The logits Z (+ bias) and values C of 8 channels of one row.
__device__ __forceinline__ void load_row(const uint16_t* C, const uint16_t* Z, const uint16_t* bias, float (&logit)[8],
                                         float (&c)[8]) {
  using V = Bf16Vec<8>;
  V::unpack(__ldg(reinterpret_cast<const uint4*>(Z)), logit);
  V::unpack(__ldg(reinterpret_cast<const uint4*>(C)), c);
  if (bias) {
    float bv[8];
    V::unpack(__ldg(reinterpret_cast<const uint4*>(bias)), bv);
#pragma unroll
    for (int j = 0; j < 8; ++j) logit[j] += bv[j];
  }
}

__device__ __forceinline__ void group0_sync() { asm volatile("bar.sync 1, 64;" ::: "memory"); }

__global__ void __launch_bounds__(kGroupThreads * kRowGroups, CSA_HCA_CTAS_PER_SM) compress_single_kernel(const CompressArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* ring_c = reinterpret_cast<uint16_t*>(smem);                   // [kStages][kStageRows][kDim]
  uint16_t* ring_z = ring_c + kStages * kStageRows * kDim;                // [kStages][kStageRows][kDim]
  uint64_t* bar = reinterpret_cast<uint64_t*>(ring_z + kStages * kStageRows * kDim);
  float* part = reinterpret_cast<float*>(smem);  // after the rows: groups 1..3's (max, sum, weighted sum)
  __shared__ float red[kGroupThreads / 32];
  pdl_launch_dependents();
  const int g = threadIdx.x / kGroupThreads, t = threadIdx.x % kGroupThreads, d0 = 8 * t;
  const int b = blockIdx.y;
  const int64_t e = blockIdx.x, i = a.entry0 + e;
  const int m = a.m;
  const int rows = m < kStageRows ? m : kStageRows;  // rows per stage (m is a power of two)
  const int stages = m / rows;
  const uint32_t bytes = static_cast<uint32_t>(rows) * kDim * 2;
  const int64_t row0 = (static_cast<int64_t>(b) * m * a.n_new + static_cast<int64_t>(m) * e) * kDim;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  auto issue = [&](int slot, int j) {  // rows j*rows .. of the block: contiguous runs of C and of Z
    mbar_arrive_expect_tx(&bar[slot], 2 * bytes);
    const int64_t off = row0 + static_cast<int64_t>(j) * rows * kDim;
    bulk_load(ring_c + slot * kStageRows * kDim, a.Ca + off, bytes, &bar[slot]);
    bulk_load(ring_z + slot * kStageRows * kDim, a.Za + off, bytes, &bar[slot]);
  };
  if (threadIdx.x == 0)
    for (int s = 0; s < kStages && s < stages; ++s) issue(s, s);
  float mx[8], den[8], num[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mx[j] = -INFINITY, den[j] = 0.f, num[j] = 0.f;
  // the slot biases of this thread's rows (at most kStageRows / kRowGroups =
  // 2 a stage), loaded one stage ahead so that no stage waits for them
  constexpr int kMine = kStageRows / kRowGroups;
  static_assert(kMine == 2, "two rows of a stage per group");
  uint4 bcur[kMine], bnext[kMine];
  auto load_bias = [&](int j, uint4 (&bv)[kMine]) {
#pragma unroll
    for (int u = 0; u < kMine; ++u) {
      const int rr = g + kRowGroups * u;
      bv[u] = (a.Ba && rr < rows && j < stages)
                  ? __ldg(reinterpret_cast<const uint4*>(a.Ba + (j * rows + rr) * kDim + d0))
                  : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load_bias(0, bnext);
  bool ok = true;
  for (int j = 0; j < stages; ++j) {
    const int slot = j % kStages;
#pragma unroll
    for (int u = 0; u < kMine; ++u) bcur[u] = bnext[u];
    load_bias(j + 1, bnext);
    ok = __syncthreads_and(mbar_wait_sleep(&bar[slot], static_cast<uint32_t>(j / kStages) & 1u, a.status)) && ok;
    {
      // this thread's two rows of the stage (rows g and g + 4), or the one
      // of them that exists when the block has fewer than 8 rows
      float logit[kMine][8], c[kMine][8];
      using V = Bf16Vec<8>;
#pragma unroll
      for (int u = 0; u < kMine; ++u) {
        const int rr = g + kRowGroups * u < rows ? g + kRowGroups * u : g;
        float bv[8];
        V::unpack(*reinterpret_cast<const uint4*>(ring_z + (slot * kStageRows + rr) * kDim + d0), logit[u]);
        V::unpack(*reinterpret_cast<const uint4*>(ring_c + (slot * kStageRows + rr) * kDim + d0), c[u]);
        V::unpack(bcur[u], bv);  // (zero without a bias)
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
          const float2 lb = __fadd2_rn(make_float2(logit[u][q], logit[u][q + 1]), make_float2(bv[q], bv[q + 1]));
          logit[u][q] = lb.x;
          logit[u][q + 1] = lb.y;
        }
      }
      if (g + kRowGroups < rows)
        online_add2(logit[0], c[0], logit[1], c[1], mx, den, num);
      else if (g < rows)
        online_add(logit[0], c[0], mx, den, num);
    }
    __syncthreads();  // the slot is read
    if (threadIdx.x == 0 && j + kStages < stages) issue(slot, j + kStages);
  }
  if (!ok && threadIdx.x == 0)  // no copy of ours stays in flight
    for (int j = stages > kStages ? stages - kStages : 0; j < stages; ++j)
      mbar_wait(&bar[j % kStages], static_cast<uint32_t>(j / kStages) & 1u, a.status);
  if (g > 0) {  // (the ring is free: every stage has been read)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      part[((g - 1) * 3 + 0) * kDim + d0 + j] = mx[j];
      part[((g - 1) * 3 + 1) * kDim + d0 + j] = den[j];
      part[((g - 1) * 3 + 2) * kDim + d0 + j] = num[j];
    }
  }
  __syncthreads();
  if (g > 0) return;
  // group 0 has at least one row (m >= 1), so its maximum is finite
#pragma unroll
  for (int h = 0; h < kRowGroups - 1; ++h) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float mh = part[(h * 3 + 0) * kDim + d0 + j];
      const float nm = fmaxf(mx[j], mh);
      const float s0 = ex2_approx((mx[j] - nm) * kLog2e), s1 = ex2_approx((mh - nm) * kLog2e);  // s1 = 0: no rows
      num[j] = fmaf(num[j], s0, part[(h * 3 + 2) * kDim + d0 + j] * s1);
      den[j] = fmaf(den[j], s0, part[(h * 3 + 1) * kDim + d0 + j] * s1);
      mx[j] = nm;
    }
  }
  float x[8], w[8], y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = __fdividef(num[j], den[j]);
  Bf16Vec<8>::unpack(__ldg(reinterpret_cast<const uint4*>(a.rms_w + d0)), w);
  norm_rope<8, kDim>(a, x, w, t, static_cast<int64_t>(m) * i, red, [] { group0_sync(); }, y);
  *reinterpret_cast<uint4*>(a.kv_out + static_cast<int64_t>(b) * a.kv_stride_b + i * kDim + d0) =
      Bf16Vec<8>::pack(y);
}

// state: [B][3][kDim] fp32 (max, sum, weighted sum of the block's tokens so far).
__global__ void __launch_bounds__(kGroupThreads) compress_single_step_kernel(const CompressArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[kGroupThreads / 32];
  const int b = blockIdx.x, t = threadIdx.x, d0 = 8 * t;
  const int64_t tp = a.q_pos[b];
  if (tp < 0) return;
  const int m = a.m;
  const int r = static_cast<int>(tp % m);  // the token's slot in its block
  float logit[8], c[8];
  load_row(a.Ca + static_cast<int64_t>(b) * kDim + d0, a.Za + static_cast<int64_t>(b) * kDim + d0,
           a.Ba ? a.Ba + r * kDim + d0 : nullptr, logit, c);
  float* st = a.state + static_cast<int64_t>(b) * 3 * kDim + d0;
  float mx[8], den[8], num[8];
  if (r == 0) {  // a block starts: the state is this token alone
#pragma unroll
    for (int j = 0; j < 8; ++j) mx[j] = logit[j], den[j] = 1.f, num[j] = c[j];
  } else {
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const float4 m4 = reinterpret_cast<const float4*>(st)[v];
      const float4 s4 = reinterpret_cast<const float4*>(st + kDim)[v];
      const float4 n4 = reinterpret_cast<const float4*>(st + 2 * kDim)[v];
      mx[4 * v] = m4.x, mx[4 * v + 1] = m4.y, mx[4 * v + 2] = m4.z, mx[4 * v + 3] = m4.w;
      den[4 * v] = s4.x, den[4 * v + 1] = s4.y, den[4 * v + 2] = s4.z, den[4 * v + 3] = s4.w;
      num[4 * v] = n4.x, num[4 * v + 1] = n4.y, num[4 * v + 2] = n4.z, num[4 * v + 3] = n4.w;
    }
    online_add(logit, c, mx, den, num);
  }
  if (r < m - 1) {  // the block goes on: keep the state
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      reinterpret_cast<float4*>(st)[v] = make_float4(mx[4 * v], mx[4 * v + 1], mx[4 * v + 2], mx[4 * v + 3]);
      reinterpret_cast<float4*>(st + kDim)[v] =
          make_float4(den[4 * v], den[4 * v + 1], den[4 * v + 2], den[4 * v + 3]);
      reinterpret_cast<float4*>(st + 2 * kDim)[v] =
          make_float4(num[4 * v], num[4 * v + 1], num[4 * v + 2], num[4 * v + 3]);
    }
    return;
  }
  const int64_t i = (tp + 1) / m - 1;  // the block is complete: entry i
  if (i >= a.n_cap) {
    if (t == 0) record_error(a.status, kErrIndexRange);
    return;
  }
  float x[8], w[8], y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = __fdividef(num[j], den[j]);
  Bf16Vec<8>::unpack(__ldg(reinterpret_cast<const uint4*>(a.rms_w + d0)), w);
  norm_rope<8, kDim>(a, x, w, t, static_cast<int64_t>(m) * i, red, [] { __syncthreads(); }, y);
  *reinterpret_cast<uint4*>(a.kv_out + static_cast<int64_t>(b) * a.kv_stride_b + i * kDim + d0) =
      Bf16Vec<8>::pack(y);
}

}  // namespace

cudaError_t launch_compress_single(const CompressArgs& args, cudaStream_t stream) {
  if (args.B <= 0) return cudaSuccess;
  if (args.m < 1 || args.m > kMaxSingleM) return cudaErrorInvalidValue;
  CompressArgs a = args;
  fill_rope(&a);
  if (a.mode == 0) {
    if (a.n_new <= 0) return cudaSuccess;
    const cudaError_t err = cudaFuncSetAttribute(compress_single_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kBulkSmem));
    if (err != cudaSuccess) return err;
    return launch_pdl(compress_single_kernel, dim3(static_cast<unsigned>(a.n_new), static_cast<unsigned>(a.B)),
                      dim3(kGroupThreads * kRowGroups), kBulkSmem, stream, a);
  }
  if (!a.state || !a.q_pos) return cudaErrorInvalidValue;
  return launch_pdl(compress_single_step_kernel, dim3(static_cast<unsigned>(a.B)), dim3(kGroupThreads), 0, stream, a);
}

}  // namespace csa
