// Shared-KV sparse MQA with a joint softmax over [window rows || selected
// compressed rows || sink].  Page "CSA / HCA" (zdszero, hca_csa), section
// "设计：近处看原文，远处看摘要" (o_{t,i} equation; the sink enters the shared
// denominator only); gather semantics "DeepSeek-V4 的 KV 压缩：从删 token 误解到
// 预算检索" §9.5–9.6; flash-style running max / running sum with a fused sink
// ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §19.3).
//
// One CTA of 8 warps per query (or per half of the heads, below).  The 64
// heads share every K=V row, so both products run with the gathered rows on
// the MMA's M side:
//   S^T[row, head]  = KV_tile[128 x 512] . Q^T[512 x 64]   (K-major A and B)
//   O^T[ch, head]  += V^T[512 x 128] . P^T[128 x 64]       (MN-major A and B)
// The same 128-byte-swizzled KV tile in shared memory serves as the K-major A
// operand of the first product and the MN-major A operand of the second.  S^T
// (64 TMEM columns) and O^T (4 x 64 columns, one per 128-channel block) live in
// TMEM.  Two warps share each TMEM lane quadrant (32 tile rows) and split the
// CTA's heads between them: a thread owns one tile row and half the heads,
// reads their logits with one tcgen05.ld, and per-head maxima and sums over
// rows use a warp reduce-scatter plus a 4-quadrant combine in shared memory.
// The reference maximum only moves when a tile exceeds it by more than 2^8,
// so O^T is rarely rescaled; the final division uses the same reference, so
// the result does not depend on when it moved.
//
// Decode (few queries) runs NH = 32 heads per CTA, two CTAs per query, so
// twice as many SMs share the per-query work; prefill runs all 64 heads per
// CTA (its rows then cross L2 once per query).  At start every CTA asks L2 to
// prefetch all of its query's rows (cp.async.bulk.prefetch.L2), so the HBM
// reads of the whole batch are in flight at once and the tile gathers that
// follow mostly hit L2.  With NH = 32 the P tile keeps its 64-head layout with
// the upper 32 columns zero, so both MMAs use the same operand layouts.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kThreads = 256;  // 8 warps: two per TMEM lane quadrant
constexpr int kTileRows = 128;
constexpr uint32_t kKVBytes = kTileRows * kDim * 2;       // 128 KiB: [8 blocks][128 rows][128 B]
constexpr uint32_t kPBytes = kTileRows * kHeads * 2;      // 16 KiB: [128 rows][64 heads]
constexpr uint32_t kKVBlock = kTileRows * 128;            // 16 KiB per 64-channel block of KV
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 64;                            // O^T columns start here
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleSlack = 8.0f;                     // log2 units

template <int NH>
constexpr size_t smem_bytes() {
  return 1024 + NH * kDim * 2 + kKVBytes + kPBytes + kMaxTopk * 4 + kTileRows * 8 + 4 * kHeads * 4 +
         4 * kHeads * 4 + 64;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled block.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Reduce-scatter of N (16 or 32) per-thread values across a warp: afterwards
// lane l holds in v[0] the reduction over all 32 lanes of value l >> (5 -
// log2 N) (lanes that share that index hold the same result).
template <int N, bool kMax>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[N]) {
  const int lane = threadIdx.x & 31;
  constexpr int kSteps = N == 32 ? 5 : 4;  // log2 N
#pragma unroll
  for (int step = 0; step < kSteps; ++step) {
    const int half = (N / 2) >> step;
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
#pragma unroll
  for (int mask = 16 >> kSteps; mask > 0; mask >>= 1) {
    const float recv = __shfl_xor_sync(0xffffffffu, v[0], mask);
    v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
  }
}

template <int NH>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(const AttnArgs a) {
  constexpr int kSplit = kHeads / NH;            // CTAs per query
  constexpr uint32_t kQBlock = NH * 128;         // bytes of one 64-channel block of Q
  constexpr int HW = NH / 2;                     // heads per warp (two warps share a TMEM quadrant)
  constexpr int kShift = HW == 32 ? 0 : 1;       // lane -> head after a reduce-scatter of HW values
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = base;                                          // [8 blocks][NH heads][128 B]
  uint8_t* kv_s = q_s + NH * kDim * 2;                          // [8 blocks][128 rows][128 B]
  uint8_t* p_s = kv_s + kKVBytes;                               // [128 rows][64 heads] bf16
  int32_t* sel_s = reinterpret_cast<int32_t*>(p_s + kPBytes);
  const uint16_t** row_src = reinterpret_cast<const uint16_t**>(sel_s + kMaxTopk);  // [128]
  float* red_s = reinterpret_cast<float*>(row_src + kTileRows);  // [4 row quadrants][NH]
  float* m_ref = red_s + 4 * kHeads;                             // running reference max (log2 units)
  float* l_sum = m_ref + kHeads;                                 // running denominator
  float* alpha = l_sum + kHeads;                                 // per-tile rescale factor
  float* fin = alpha + kHeads;                                   // final per-head output scale
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(fin + kHeads);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);            // [0] n_sel, [1] rescale

  pdl_launch_dependents();
  pdl_wait();  // before any global access and before TMEM is taken
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;                  // TMEM lane quadrant == 32 tile rows
  const int hw0 = (warp >> 2) * HW;           // first head (within the CTA) of this warp
  const int qi = blockIdx.x / kSplit;
  const int h0 = (blockIdx.x % kSplit) * NH;  // first head of this CTA
  const int b = blockIdx.y;
  const int64_t row_q = static_cast<int64_t>(b) * a.Q + qi;
  const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[row_q]) : a.pos_base + qi;

  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  if (tid == 0) {
    mbar_init(mma_bar, 1);
    fence_mbar_init();
    flags[1] = 0;
  }
  if (tid < NH) {
    m_ref[tid] = -INFINITY;
    l_sum[tid] = 0.f;
  }

  // Q tile of this CTA's heads: [8 channel blocks][NH heads][128 B], swizzled.
  {
    const uint16_t* qg = a.q + (row_q * kHeads + h0) * kDim;
    for (int ch = tid; ch < NH * kDim / 8; ch += kThreads) {
      const int h = ch >> 6, blk = (ch >> 3) & 7, c = ch & 7;
      cp_async_16(q_s + blk * kQBlock + swz(h, c), qg + h * kDim + blk * 64 + c * 8);
    }
  }
  if (NH < 64) {  // the P tile's unused head columns stay zero
    for (int r = tid; r < kTileRows; r += kThreads)
#pragma unroll
      for (int c = NH / 8; c < 8; ++c) *reinterpret_cast<uint4*>(p_s + swz(r, c)) = make_uint4(0u, 0u, 0u, 0u);
  }

  // Compact the selected entries (drop -1, flag out-of-range indices).
  {
    const int32_t* ig = a.idx + row_q * a.k;
    const int per = (a.k + kThreads - 1) / kThreads;
    const int lo = min(a.k, tid * per), hi = min(a.k, lo + per);
    int cnt = 0;
    for (int j = lo; j < hi; ++j) {
      const int32_t v = ig[j];
      if (v >= 0 && v < a.n_cap) ++cnt;
      else if (v != -1 && h0 == 0) record_error(a.status, kErrIndexRange);
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
    for (int j = lo; j < hi; ++j) {
      const int32_t v = ig[j];
      if (v >= 0 && v < a.n_cap) sel_s[before++] = v;
    }
    if (tid == kThreads - 1) flags[0] = before;
  }
  cp_async_commit_wait_all();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tlane = tmem + (static_cast<uint32_t>(quad * 32) << 16);  // this warp's TMEM quadrant
  const int n_sel = flags[0];
  const int n_swa = static_cast<int>(t < 0 ? 0 : min(static_cast<int64_t>(a.W), t + 1));
  const int n_rows = n_swa + n_sel;
  const int n_tiles = (n_rows + kTileRows - 1) / kTileRows;
  const float scale2 = a.sm_scale * kLog2e;
  const uint16_t* kv_b = a.kv + static_cast<int64_t>(b) * a.n_cap * kDim;
  const int64_t swa_pos0 = a.swa_mode == 1 ? (a.swa_pos0 ? a.swa_pos0[b] : a.swa_pos0_base) : 0;

  // Address of row j of this query's row set (null: absent / skipped).
  auto row_at = [&](int j) -> const uint16_t* {
    if (j < n_swa) {
      const int64_t u = t - n_swa + 1 + j;  // window position
      if (a.swa_mode == 0) return a.swa + (static_cast<int64_t>(b) * a.W + u % a.W) * kDim;
      const int64_t rr = u - swa_pos0;
      if (rr >= 0 && rr < a.swa_len) return a.swa + (static_cast<int64_t>(b) * a.swa_len + rr) * kDim;
      return nullptr;
    }
    if (j < n_rows) return kv_b + static_cast<int64_t>(sel_s[j - n_swa]) * kDim;
    return nullptr;
  };
  // Put every row of this query in flight towards L2 now.
  for (int j = tid; j < n_rows; j += kThreads) {
    const uint16_t* src = row_at(j);
    if (src) prefetch_l2(src, kDim * 2);
  }

  constexpr uint32_t idesc_s = instr_desc(kTileRows, NH, 1, 1, 0, 0);      // bf16, K-major A/B
  constexpr uint32_t idesc_o = instr_desc(kTileRows, kHeads, 1, 1, 1, 1);  // bf16, MN-major A/B
  uint32_t phase = 0;
  bool ok = true;

  for (int tile = 0; tile < n_tiles && ok; ++tile) {
    const int r0 = tile * kTileRows;
    // ---- resolve the tile's 128 row addresses
    if (tid < kTileRows) {
      const int j = r0 + tid;
      const uint16_t* src = row_at(j);
      if (!src && j < n_swa && h0 == 0) record_error(a.status, kErrIndexRange);
      row_src[tid] = src;
    }
    __syncthreads();
    // ---- gather 128 rows (16-byte cp.async, a warp covers 512 contiguous bytes)
    for (int ch = tid; ch < kTileRows * 64; ch += kThreads) {
      const int r = ch >> 6, blk = (ch >> 3) & 7, c = ch & 7;
      const uint16_t* src = row_src[r];
      uint8_t* dst = kv_s + blk * kKVBlock + swz(r, c);
      if (src) cp_async_16(dst, src + blk * 64 + c * 8);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_commit_wait_all();
    fence_proxy_async_smem();
    __syncthreads();

    // ---- S^T = KV . Q^T  (32 MMAs of K = 16)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kvb = smem_u32(kv_s), qb = smem_u32(q_s);
#pragma unroll
      for (int blk = 0; blk < 8; ++blk)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = smem_desc(kvb + blk * kKVBlock + kk * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(qb + blk * kQBlock + kk * 32, 16, 1024, kSwizzle128B);
          mma_f16(tmem, ad, bd, idesc_s, (blk | kk) ? 1u : 0u);
        }
      tc_commit(mma_bar);
    }
    __syncwarp();
    // block-uniform: every thread waits, all leave together if one gave up
    if (!__syncthreads_and(mbar_wait(mma_bar, phase, a.status))) { ok = false; break; }
    phase ^= 1u;
    tc_fence_after();

    // ---- logits of this thread's row (its warp's HW heads), per-head tile max
    const int r = quad * 32 + lane;  // TMEM lane == tile row
    const bool valid = row_src[r] != nullptr;
    float l[HW];
    {
      if constexpr (HW == 32) {
        uint32_t v[32];
        tmem_ld32(tlane + hw0, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; ++h) l[h] = valid ? __uint_as_float(v[h]) * scale2 : -INFINITY;
      } else {
        uint32_t v[16];
        tmem_ld16(tlane + hw0, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h) l[h] = valid ? __uint_as_float(v[h]) * scale2 : -INFINITY;
      }
    }
    {
      float tmp[HW];
#pragma unroll
      for (int h = 0; h < HW; ++h) tmp[h] = l[h];
      warp_reduce_scatter<HW, true>(tmp);
      if ((lane & kShift) == 0) red_s[quad * NH + hw0 + (lane >> kShift)] = tmp[0];
    }
    __syncthreads();
    if (tid < NH) {
      const float tmax = fmaxf(fmaxf(red_s[tid], red_s[NH + tid]), fmaxf(red_s[2 * NH + tid], red_s[3 * NH + tid]));
      const float mo = m_ref[tid];
      float al = 1.f;
      if (tmax > mo + kRescaleSlack) {  // also taken on the first tile (mo = -inf)
        al = (mo == -INFINITY) ? 0.f : exp2f(mo - tmax);
        m_ref[tid] = tmax;
        l_sum[tid] *= al;
        if (tile > 0 && al != 1.f) flags[1] = 1;
      }
      alpha[tid] = al;
    }
    __syncthreads();

    // ---- rescale the O^T columns of this warp's heads when a reference moved
    if (flags[1]) {
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        const uint32_t taddr = tlane + kOCol + blk * 64 + hw0;
        if constexpr (HW == 32) {
          uint32_t v[32];
          tmem_ld32(taddr, v);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] = __float_as_uint(__uint_as_float(v[h]) * alpha[hw0 + h]);
          tmem_st32(taddr, v);
        } else {
          uint32_t v[16];
          tmem_ld16(taddr, v);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) v[h] = __float_as_uint(__uint_as_float(v[h]) * alpha[hw0 + h]);
          tmem_st16(taddr, v);
        }
      }
      tmem_wait_st();
    }

    // ---- P = 2^(l - m_ref) as bf16 into the swizzled P tile; row sums
    {
      float pf[HW];
#pragma unroll
      for (int c = 0; c < HW / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = c * 8 + 2 * i;
          const float m0 = m_ref[hw0 + h], m1 = m_ref[hw0 + h + 1];
          const float ref0 = m0 == -INFINITY ? 0.f : m0;
          const float ref1 = m1 == -INFINITY ? 0.f : m1;
          const __nv_bfloat162 pb = __floats2bfloat162_rn(exp2f(l[h] - ref0), exp2f(l[h + 1] - ref1));
          pf[h] = __low2float(pb);
          pf[h + 1] = __high2float(pb);
          w[i] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        *reinterpret_cast<uint4*>(p_s + swz(r, hw0 / 8 + c)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      warp_reduce_scatter<HW, false>(pf);
      __syncthreads();  // everyone is done reading red_s (tile max) and flags
      if ((lane & kShift) == 0) red_s[quad * NH + hw0 + (lane >> kShift)] = pf[0];
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid < NH) {
      l_sum[tid] += (red_s[tid] + red_s[NH + tid]) + (red_s[2 * NH + tid] + red_s[3 * NH + tid]);
      if (tid == 0) flags[1] = 0;
    }

    // ---- O^T += V^T . P^T  (4 channel blocks x 8 K-steps of 16 rows)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kvb = smem_u32(kv_s), pb = smem_u32(p_s);
#pragma unroll
      for (int blk = 0; blk < 4; ++blk)
#pragma unroll
        for (int ks = 0; ks < kTileRows / 16; ++ks) {
          const uint64_t ad = smem_desc(kvb + 2 * blk * kKVBlock + ks * 2048, kKVBlock, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(pb + ks * 2048, kPBytes, 1024, kSwizzle128B);
          mma_f16(tmem + kOCol + blk * 64, ad, bd, idesc_o, (tile > 0 || ks > 0) ? 1u : 0u);
        }
      tc_commit(mma_bar);
    }
    __syncwarp();
    if (!__syncthreads_and(mbar_wait(mma_bar, phase, a.status))) { ok = false; break; }
    phase ^= 1u;
    tc_fence_after();
    __syncthreads();  // kv_s / p_s may be overwritten by the next tile
  }

  // ---- epilogue: out = O^T / (l_sum + 2^(sink*log2e - m_ref))
  __syncthreads();
  if (tid < NH) {
    const float mr = m_ref[tid];
    const float sk = a.sink[h0 + tid] * kLog2e;
    const float M = fmaxf(mr, sk);
    const float keep = mr == -INFINITY ? 0.f : exp2f(mr - M);
    const float den = l_sum[tid] * keep + exp2f(sk - M);
    fin[tid] = M == -INFINITY ? 0.f : keep / den;
    if (a.lse) a.lse[row_q * kHeads + h0 + tid] = M == -INFINITY ? -INFINITY : (M + log2f(den)) / kLog2e;
  }
  __syncthreads();
  uint16_t* out_s = reinterpret_cast<uint16_t*>(kv_s);  // [NH heads][512] bf16 staging
  if (ok && n_tiles > 0) {
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      const int chn = blk * 128 + quad * 32 + lane;
      const uint32_t taddr = tlane + kOCol + blk * 64 + hw0;
      if constexpr (HW == 32) {
        uint32_t v[32];
        tmem_ld32(taddr, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; ++h)
          out_s[(hw0 + h) * kDim + chn] =
              __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[h]) * fin[hw0 + h]));
      } else {
        uint32_t v[16];
        tmem_ld16(taddr, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h)
          out_s[(hw0 + h) * kDim + chn] =
              __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[h]) * fin[hw0 + h]));
      }
    }
  } else {
    for (int e = tid; e < NH * kDim; e += kThreads) out_s[e] = 0;
  }
  __syncthreads();
  {
    uint4* og = reinterpret_cast<uint4*>(a.out + (row_q * kHeads + h0) * kDim);
    const uint4* os = reinterpret_cast<const uint4*>(out_s);
    for (int e = tid; e < NH * kDim / 8; e += kThreads) og[e] = os[e];
  }

  // A timed-out wait leaves MMAs possibly in flight: give them a bounded
  // chance to finish before TMEM is released.
  if (!ok && tid == 0) mbar_wait(mma_bar, phase, a.status);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NH>
cudaError_t launch_nh(const AttnArgs& a, cudaStream_t stream) {
  constexpr size_t smem = smem_bytes<NH>();
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(sparse_attn_kernel<NH>, dim3(a.Q * (kHeads / NH), a.B), dim3(kThreads), smem, stream, a);
}

}  // namespace

cudaError_t launch_sparse_attn(const AttnArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode, cudaStream_t stream) {
  (void)encode;  // rows are gathered with cp.async; no tensor map is needed
  if (a.B <= 0 || a.Q <= 0) return cudaSuccess;
  // Few queries: split the heads over two CTAs per query to occupy more SMs.
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (static_cast<int64_t>(a.B) * a.Q < sms) return launch_nh<32>(a, stream);
  return launch_nh<64>(a, stream);
}

}  // namespace csa
