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
// Warp roles (192 threads):
//   warp 0      TMA producer: q^I once, then a STAGES-deep ring of 16 KiB
//               K^I tiles (128-byte swizzle), L2 evict-first;
//   warp 1      TMEM owner and MMA issuer (one thread), double-buffered
//               accumulators so the epilogue of tile n overlaps MMA n+1;
//   warps 2..5  epilogue: tcgen05.ld, weighted ReLU sum, coalesced fp32
//               score stores (only for keys visible to the query).
// Every wait is bounded; a timeout records the error, the roles drain their
// own in-flight work and the CTA releases TMEM and exits.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kTileKeys = 128;
constexpr uint32_t kKeyTileBytes = kTileKeys * kIdxDim;   // 16 KiB
constexpr uint32_t kQBytes = kIdxHeads * kIdxDim;         // 8 KiB per query

template <int QPC>
struct IndexCfg {
  static constexpr int N = kIdxHeads * QPC;
  static constexpr int STAGES = QPC == 1 ? 6 : 6;
  static constexpr uint32_t TMEM_COLS = 2 * N;
  static constexpr size_t SMEM = 1024 + QPC * kQBytes + STAGES * kKeyTileBytes + QPC * kIdxHeads * 4 +
                                 (2 * STAGES + 6) * 8 + 16 + QPC * 8 + 16;
};

template <int QPC>
__global__ void __launch_bounds__(192, 1)
    index_score_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                       const IndexArgs a, const int tiles_per_cta) {
  using Cfg = IndexCfg<QPC>;
  constexpr int N = Cfg::N;
  constexpr int STAGES = Cfg::STAGES;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = base;
  uint8_t* k_s = q_s + QPC * kQBytes;
  float* w_s = reinterpret_cast<float*>(k_s + STAGES * kKeyTileBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(w_s + QPC * kIdxHeads);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* q_full = acc_empty + 2;
  uint64_t* mma_done = q_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int64_t* vis = reinterpret_cast<int64_t*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int q0 = blockIdx.y * QPC;

  // Visible entries V(t) = floor((t+1)/m) of each query of the group.
  if (threadIdx.x < QPC) {
    const int q = q0 + threadIdx.x;
    int64_t V = 0;
    if (q < a.Q) {
      const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[static_cast<int64_t>(b) * a.Q + q]) : a.pos_base + q;
      V = t >= 0 ? (t + 1) / a.m : 0;
      if (V > a.n_cap) {
        if (blockIdx.x == 0) record_error(a.status, kErrIndexRange);
        V = a.n_cap;
      }
    }
    vis[threadIdx.x] = V;
  }
  __syncthreads();
  int64_t vmax = 0;
#pragma unroll
  for (int j = 0; j < QPC; ++j) vmax = vis[j] > vmax ? vis[j] : vmax;
  const int64_t tile0 = static_cast<int64_t>(blockIdx.x) * tiles_per_cta;
  const int64_t tiles_needed = (vmax + kTileKeys - 1) / kTileKeys;
  const int n_my = static_cast<int>(min(static_cast<int64_t>(tiles_per_cta), tiles_needed - tile0));
  if (n_my <= 0) return;  // uniform: nothing of this group is visible here

  if (warp == 1) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&acc_full[x], 1);
      mbar_init(&acc_empty[x], 4);
    }
    mbar_init(q_full, 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (threadIdx.x >= 64) {
    for (int e = threadIdx.x - 64; e < QPC * kIdxHeads; e += 128) {
      const int q = q0 + e / kIdxHeads;
      const int h = e % kIdxHeads;
      const uint16_t wb = q < a.Q ? a.wI[(static_cast<int64_t>(b) * a.Q + q) * kIdxHeads + h] : uint16_t(0);
      w_s[e] = __uint_as_float(static_cast<uint32_t>(wb) << 16);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_q);
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(q_full, QPC * kQBytes);
      for (int j = 0; j < QPC; ++j)
        tma_load_2d(q_s + j * kQBytes, &tm_q, 0,
                    static_cast<int32_t>((static_cast<int64_t>(b) * a.Q + q0 + j) * kIdxHeads), q_full);
      uint32_t issued = 0, parity = 0;
      for (int it = 0; it < n_my; ++it) {
        const int s = it % STAGES;
        const uint32_t use = static_cast<uint32_t>(it / STAGES);
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1u, a.status)) break;
        mbar_arrive_expect_tx(&full[s], kKeyTileBytes);
        tma_load_3d(k_s + s * kKeyTileBytes, &tm_k, 0, static_cast<int32_t>((tile0 + it) * kTileKeys), b,
                    &full[s], pol);
        issued |= 1u << s;
        parity = (parity & ~(1u << s)) | ((use & 1u) << s);
      }
      // Our own copies must have landed before the CTA may exit.
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) mbar_wait(&full[s], (parity >> s) & 1u, a.status);
      mbar_wait(q_full, 0, a.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(kTileKeys, N, 0, 0, 0, 0);
      bool ok = mbar_wait(q_full, 0, a.status);
      const uint32_t qb = smem_u32(q_s);
      for (int it = 0; ok && it < n_my; ++it) {
        const int s = it % STAGES;
        const uint32_t use = static_cast<uint32_t>(it / STAGES);
        const int x = it & 1;
        const uint32_t xuse = static_cast<uint32_t>(it >> 1);
        if (xuse > 0 && !(ok = mbar_wait(&acc_empty[x], (xuse - 1) & 1u, a.status))) break;
        if (!(ok = mbar_wait(&full[s], use & 1u, a.status))) break;
        tc_fence_after();
        const uint32_t kb = smem_u32(k_s + s * kKeyTileBytes);
#pragma unroll
        for (int kk = 0; kk < kIdxDim / 32; ++kk) {
          const uint64_t ad = smem_desc(kb + kk * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(qb + kk * 32, 16, 1024, kSwizzle128B);
          mma_f8(tmem + x * N, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        tc_commit(&empty[s]);
        tc_commit(&acc_full[x]);
      }
      tc_commit(mma_done);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue ----------------
    const int sub = warp & 3;  // TMEM sub-partition this warp may access
    const int row = sub * 32 + lane;
    for (int it = 0; it < n_my; ++it) {
      const int x = it & 1;
      const uint32_t xuse = static_cast<uint32_t>(it >> 1);
      // every lane waits; the warp leaves together if any lane gave up
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[x], xuse & 1u, a.status))) break;
      tc_fence_after();
      const int64_t s_idx = (tile0 + it) * kTileKeys + row;
#pragma unroll
      for (int j = 0; j < QPC; ++j) {
        uint32_t r0[32], r1[32];
        const uint32_t taddr = tmem + (static_cast<uint32_t>(sub * 32) << 16) + x * N + j * kIdxHeads;
        tmem_ld32(taddr, r0);
        tmem_ld32(taddr + 32, r1);
        tmem_wait_ld();
        const float* w = w_s + j * kIdxHeads;
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < 32; ++h) acc = fmaf(w[h], fmaxf(__uint_as_float(r0[h]), 0.f), acc);
#pragma unroll
        for (int h = 0; h < 32; ++h) acc = fmaf(w[32 + h], fmaxf(__uint_as_float(r1[h]), 0.f), acc);
        if (s_idx < vis[j]) a.scores[(static_cast<int64_t>(b) * a.Q + q0 + j) * a.score_ld + s_idx] = acc;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[x]);
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

bool encode_maps(const IndexArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode, int qpc, CUtensorMap* tm_k,
                 CUtensorMap* tm_q) {
  // K^I: [B][n_cap][128] bytes, box = 128 keys x 128 bytes of one sequence.
  cuuint64_t kdim[3] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(a.n_cap),
                        static_cast<cuuint64_t>(a.B)};
  cuuint64_t kstride[2] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(a.n_cap) * kIdxDim};
  cuuint32_t kbox[3] = {static_cast<cuuint32_t>(kIdxDim), static_cast<cuuint32_t>(kTileKeys), 1};
  cuuint32_t ones[3] = {1, 1, 1};
  if (encode(tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.kI), kdim, kstride, kbox, ones,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  // q^I: [B*Q*64 rows][128 bytes], box = the 64 heads of one query.
  cuuint64_t qdim[2] = {static_cast<cuuint64_t>(kIdxDim),
                        static_cast<cuuint64_t>(a.B) * static_cast<cuuint64_t>(a.Q) * kIdxHeads};
  cuuint64_t qstride[1] = {static_cast<cuuint64_t>(kIdxDim)};
  cuuint32_t qbox[2] = {static_cast<cuuint32_t>(kIdxDim), static_cast<cuuint32_t>(kIdxHeads)};
  (void)qpc;
  return encode(tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.qI), qdim, qstride, qbox, ones,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int QPC>
cudaError_t launch_qpc(const IndexArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode, cudaStream_t stream) {
  using Cfg = IndexCfg<QPC>;
  CUtensorMap tm_k, tm_q;
  if (!encode_maps(a, encode, QPC, &tm_k, &tm_q)) return cudaErrorInvalidValue;
  static bool attr_set = false;  // per process; the attribute is per function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(index_score_kernel<QPC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t tiles_per_seq = (a.n_cap + kTileKeys - 1) / kTileKeys;
  const int64_t groups = (a.Q + QPC - 1) / QPC;
  // Enough CTAs to cover every SM several times, with at least 4 tiles each
  // so the pipeline has room to run.
  const int64_t target_ctas = 4LL * sms;
  int64_t per_cta = (tiles_per_seq * groups * a.B + target_ctas - 1) / target_ctas;
  if (per_cta < 4) per_cta = 4;
  if (per_cta > tiles_per_seq) per_cta = tiles_per_seq;
  const int64_t chunks = (tiles_per_seq + per_cta - 1) / per_cta;
  dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(groups), static_cast<unsigned>(a.B));
  index_score_kernel<QPC><<<grid, 192, Cfg::SMEM, stream>>>(tm_k, tm_q, a, static_cast<int>(per_cta));
  return counted(cudaGetLastError());
}

}  // namespace

cudaError_t launch_index_scores(const IndexArgs& a, PFN_cuTensorMapEncodeTiled_v12000 encode,
                                cudaStream_t stream) {
  if (a.B <= 0 || a.Q <= 0) return cudaSuccess;
  if (a.Q >= 4) return launch_qpc<4>(a, encode, stream);
  return launch_qpc<1>(a, encode, stream);
}

}  // namespace csa
