// Overlapped CSA compressor for one entry: per-channel softmax pooling over
// 2m slots, RMSNorm, partial RoPE.  Page "CSA / HCA" (zdszero, hca_csa),
// section "CSA 的重叠窗口" (Softmax_row and C_i^Comp equations, i = 0
// boundary); RoPE position = first token of the entry's block ("DeepSeek-V4
// CSA/HCA 与 DeepSeek-V4.1 CSA2" §7.4); decode emission only at a block
// boundary ("DeepSeek-V4 的 KV 压缩：从删 token 误解到预算检索" §9.3).
//
// A group of kDim / CPT threads computes one entry; thread t owns channels
// CPT*t .. CPT*t+CPT-1 and reads each of the 4*m source rows it needs with
// one load of CPT bf16 values.  Softmax, normalisation and rotation are fp32;
// the RoPE angle is formed exactly as a fixed-point fraction of a turn
// (rope_sincos in kernels.h: positions reach 2^20 and beyond, where an fp32
// angle would be off by ~0.1 rad), from the 32 frequencies that come with
// the arguments, then the hardware sine and cosine per pair.  The softmax
// weights use the hardware exp2 and divide (a few ulp each: far inside the
// bf16 outputs' rounding and the FP8 key codes' midpoint band).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fp4.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace csa {

template <int CPT>
struct Bf16Vec;
template <>
struct Bf16Vec<1> {
  using T = uint16_t;
  static __device__ __forceinline__ void unpack(const T u, float (&v)[1]) {
    v[0] = __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
};
template <>
struct Bf16Vec<8> {
  using T = uint4;
  static __device__ __forceinline__ void unpack(const T u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ T pack(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Bf16Vec<4> {
  using T = uint2;
  static __device__ __forceinline__ void unpack(const T u, float (&v)[4]) {
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  }
  static __device__ __forceinline__ T pack(const float (&v)[4]) {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
  }
};
template <>
struct Bf16Vec<2> {
  using T = uint32_t;
  static __device__ __forceinline__ void unpack(const T u, float (&v)[2]) {
    v[0] = __uint_as_float(u << 16);
    v[1] = __uint_as_float(u & 0xFFFF0000u);
  }
  static __device__ __forceinline__ T pack(const float (&v)[2]) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[0], v[1]);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
};

// 2^x by the hardware approximation (a few ulp; results below 2^-126
// flush to zero, a weight that adds nothing to a sum of weights of at
// least 1).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// RMSNorm of the pooled entry x over its D channels (thread t holds channels
// CPT*t .. CPT*t+CPT-1; `red` one float per warp of the D/CPT threads, sync()
// a barrier over exactly them), times the weight w, then partial RoPE on the
// last kRope channels in interleaved pairs at position pos, into y.
template <int CPT, int D, class Sync>
__device__ __forceinline__ void norm_rope(const CompressArgs& a, const float (&x)[CPT], const float (&w)[CPT], int t,
                                          int64_t pos, float* red, Sync sync, float (&y)[CPT]) {
  constexpr int NT = D / CPT;
  const int d0 = t * CPT;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) ss = fmaf(x[j], x[j], ss);
  // warp sums, then the group's warps combine
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((t & 31) == 0) red[t >> 5] = ss;
  sync();
  float total = 0.f;
#pragma unroll
  for (int wi = 0; wi < NT / 32; ++wi) total += red[wi];
  const float inv = rsqrtf(total / static_cast<float>(D) + a.rms_eps);
#pragma unroll
  for (int j = 0; j < CPT; ++j) y[j] = x[j] * inv * w[j];

  // Partial RoPE on channels D-R .. D-1, interleaved pairs (one channel
  // per thread: the pair's other channel is the neighbouring lane's).
  if constexpr (CPT == 1) {
    const float o = __shfl_xor_sync(0xffffffffu, y[0], 1);
    if (d0 >= D - kRope) {
      float s, c;
      rope_sincos(pos, a.rope_turns[(d0 - (D - kRope)) >> 1], &s, &c);
      y[0] = (d0 & 1) ? fmaf(o, s, y[0] * c) : fmaf(y[0], c, -o * s);
    }
  } else if (d0 >= D - kRope) {
#pragma unroll
    for (int pr = 0; pr < CPT / 2; ++pr) {
      const int jp = (d0 + 2 * pr - (D - kRope)) / 2;
      float s, c;
      rope_sincos(pos, a.rope_turns[jp], &s, &c);
      const float u = y[2 * pr], v = y[2 * pr + 1];
      y[2 * pr] = u * c - v * s;
      y[2 * pr + 1] = u * s + v * c;
    }
  }
}

// The values of entry (e-th of the chunk in bulk mode; the one completing at
// q_pos[b] in ring mode) of sequence b at width D (rows of D channels, RoPE
// on the last kRope of them): thread t's channels CPT*t .. CPT*t+CPT-1 into
// y, the entry's index into *entry.  Returns false when there is no entry
// (ring mode between block boundaries, or past the cache).  `red` holds one
// float per warp of the group; sync() is a barrier over exactly the group's
// threads.  Every thread of the group must call this with the same (b, e).
// kStaged (bulk mode only): the entry's source rows are already in shared
// memory at `stage` (block i's M rows of Z, its M rows of C, then block
// i-1's Z and C rows; D channels each) and are read where they are used.
// kPrefetch (ring mode, callers with registers to spare): every slot of both
// streams, the slot biases and the weight are loaded before the position is
// read (one memory round trip, not two), and the halves are put in block
// order once it is known.
template <int M, int CPT, int D, class Sync, bool kStaged = false, bool kPrefetch = false>
__device__ bool compress_values(const CompressArgs& a, int b, int64_t e, int t, float* red, Sync sync,
                                float (&y)[CPT], int64_t* entry, const uint16_t* stage = nullptr) {
  using V = Bf16Vec<CPT>;
  using L = typename V::T;
  const int d0 = t * CPT;

  constexpr bool kAllSlots = kPrefetch && !kStaged;
  L ra_z[kAllSlots ? 2 * M : 1], ra_c[kAllSlots ? 2 * M : 1], rb_z[kAllSlots ? 2 * M : 1], rb_c[kAllSlots ? 2 * M : 1];
  L pb[kAllSlots ? 2 * M : 1], pw = {};
  if constexpr (kAllSlots) {
    if (a.mode != 0) {
      const int64_t ring = static_cast<int64_t>(b) * 2 * M * D;
#pragma unroll
      for (int s = 0; s < 2 * M; ++s) {
        ra_z[s] = __ldg(reinterpret_cast<const L*>(a.Za + ring + s * D + d0));
        ra_c[s] = __ldg(reinterpret_cast<const L*>(a.Ca + ring + s * D + d0));
        rb_z[s] = __ldg(reinterpret_cast<const L*>(a.Zb + ring + s * D + d0));
        rb_c[s] = __ldg(reinterpret_cast<const L*>(a.Cb + ring + s * D + d0));
        pb[s] = __ldg(reinterpret_cast<const L*>((s < M ? a.Ba + s * D : a.Bb + (s - M) * D) + d0));
      }
      pw = __ldg(reinterpret_cast<const L*>(a.rms_w + d0));
    }
  }

  // Locate entry i and the rows of block i (a stream) and block i-1 (b stream).
  int64_t i;
  const uint16_t *ca[M], *za[M], *cb[M], *zb[M];
  bool has_prev;
  if (a.mode == 0) {
    i = a.entry0 + e;
    has_prev = i > 0;
    const int64_t T = static_cast<int64_t>(M) * a.n_new;
    const int64_t seq = static_cast<int64_t>(b) * T * D;
#pragma unroll
    for (int r = 0; r < M; ++r) {
      const int64_t row_a = seq + (M * e + r) * D;
      ca[r] = a.Ca + row_a;
      za[r] = a.Za + row_a;
      if (e > 0) {
        const int64_t row_b = seq + (M * (e - 1) + r) * D;
        cb[r] = a.Cb + row_b;
        zb[r] = a.Zb + row_b;
      } else {
        // block entry0-1 lives in the separate "previous block" rows
        const int64_t row_b = (static_cast<int64_t>(b) * M + r) * D;
        cb[r] = a.Cb_prev ? a.Cb_prev + row_b : nullptr;
        zb[r] = a.Zb_prev ? a.Zb_prev + row_b : nullptr;
      }
    }
  } else {
    const int64_t tp = a.q_pos[b];
    if (tp < 0 || (tp + 1) % M != 0) return false;  // no block completes at this step
    i = (tp + 1) / M - 1;
    if (i >= a.n_cap) {
      if (t == 0) record_error(a.status, kErrIndexRange);
      return false;
    }
    has_prev = i > 0;
    const int64_t ring = static_cast<int64_t>(b) * 2 * M * D;
#pragma unroll
    for (int r = 0; r < M; ++r) {
      const int64_t slot_a = (M * i + r) % (2 * M);
      const int64_t slot_b = (M * (i - 1) + r + 2 * M) % (2 * M);
      ca[r] = a.Ca + ring + slot_a * D;
      za[r] = a.Za + ring + slot_a * D;
      cb[r] = a.Cb + ring + slot_b * D;
      zb[r] = a.Zb + ring + slot_b * D;
    }
  }

  // Issue every load of the entry first (one memory round trip), then math;
  // staged rows (and then the slot biases, cache-resident) are read at use.
  L zr[kStaged ? 1 : 2 * M], cr[kStaged ? 1 : 2 * M], br[kStaged ? 1 : 2 * M];
  if (kAllSlots && a.mode != 0) {  // block i holds ring slots half .. half+M-1, block i-1 the others
    const bool upper = (M * i) % (2 * M) != 0;
#pragma unroll
    for (int r = 0; r < M; ++r) {
      zr[r] = upper ? ra_z[(M + r) % (2 * M)] : ra_z[r];
      cr[r] = upper ? ra_c[(M + r) % (2 * M)] : ra_c[r];
      zr[M + r] = upper ? rb_z[r] : rb_z[(M + r) % (2 * M)];
      cr[M + r] = upper ? rb_c[r] : rb_c[(M + r) % (2 * M)];
      br[r] = pb[r];
      br[M + r] = pb[M + r];
    }
  } else if constexpr (!kStaged) {
#pragma unroll
    for (int r = 0; r < M; ++r) {
      zr[r] = __ldg(reinterpret_cast<const L*>(za[r] + d0));
      cr[r] = __ldg(reinterpret_cast<const L*>(ca[r] + d0));
      br[r] = __ldg(reinterpret_cast<const L*>(a.Ba + r * D + d0));
      if (has_prev) {
        zr[M + r] = __ldg(reinterpret_cast<const L*>(zb[r] + d0));
        cr[M + r] = __ldg(reinterpret_cast<const L*>(cb[r] + d0));
        br[M + r] = __ldg(reinterpret_cast<const L*>(a.Bb + r * D + d0));
      }
    }
  }
  const auto z_at = [&](int r) -> L {
    if constexpr (kStaged) return *reinterpret_cast<const L*>(stage + ((r < M ? 0 : 2 * M) + r % M) * D + d0);
    else return zr[r];
  };
  const auto c_at = [&](int r) -> L {
    if constexpr (kStaged) return *reinterpret_cast<const L*>(stage + ((r < M ? M : 3 * M) + r % M) * D + d0);
    else return cr[r];
  };
  const auto b_at = [&](int r) -> L {
    if constexpr (kStaged)
      return __ldg(reinterpret_cast<const L*>((r < M ? a.Ba + r * D : a.Bb + (r - M) * D) + d0));
    else return br[r];
  };
  const L wr = (kAllSlots && a.mode != 0) ? pw : __ldg(reinterpret_cast<const L*>(a.rms_w + d0));
  const int slots = has_prev ? 2 * M : M;  // block i-1 slots are absent for entry 0

  // Maximum logit (Z + B) of the slots, per channel.
  float mx[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) mx[j] = -INFINITY;
#pragma unroll
  for (int r = 0; r < 2 * M; ++r) {
    if (r < slots) {
      float z[CPT], bias[CPT];
      V::unpack(z_at(r), z);
      V::unpack(b_at(r), bias);
#pragma unroll
      for (int j = 0; j < CPT; ++j) mx[j] = fmaxf(mx[j], z[j] + bias[j]);
    }
  }

  // Softmax-weighted sum of the C rows.
  constexpr float kLog2e = 1.4426950408889634f;
  float num[CPT], den[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) num[j] = den[j] = 0.f;
#pragma unroll
  for (int r = 0; r < 2 * M; ++r) {
    if (r < slots) {
      float z[CPT], bias[CPT], c[CPT];
      V::unpack(z_at(r), z);
      V::unpack(b_at(r), bias);
      V::unpack(c_at(r), c);
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const float w = ex2_approx((z[j] + bias[j] - mx[j]) * kLog2e);
        num[j] = fmaf(w, c[j], num[j]);
        den[j] += w;
      }
    }
  }
  float x[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) x[j] = __fdividef(num[j], den[j]);  // den in [1, 2M]: the largest slot weighs 1
  float w[CPT];
  V::unpack(wr, w);
  norm_rope<CPT, D>(a, x, w, t, static_cast<int64_t>(M) * i, red, sync, y);
  *entry = i;
  return true;
}

// Entry of the main compressor (width 512), stored as bf16 into kv_out, or
// (kv_fp4_out set) as the FP4 entry of its bf16 values: a 16-channel group
// is 16/CPT adjacent threads, whose maximum is taken by shuffles.
template <int M, int CPT, class Sync, bool kStaged = false>
__device__ void compress_entry(const CompressArgs& a, int b, int64_t e, int t, float* red, Sync sync,
                               const uint16_t* stage = nullptr) {
  using V = Bf16Vec<CPT>;
  float y[CPT];
  int64_t i;
  if (!compress_values<M, CPT, kDim, Sync, kStaged>(a, b, e, t, red, sync, y, &i, stage)) return;
  if (!a.kv_fp4_out) {
    *reinterpret_cast<typename V::T*>(a.kv_out + static_cast<int64_t>(b) * a.kv_stride_b + i * kDim + t * CPT) =
        V::pack(y);
    return;
  }
  static_assert(CPT >= 2 && 16 % CPT == 0, "a group of 16 channels spans whole threads");
  constexpr int kGroupThreads = 16 / CPT;
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    y[j] = __bfloat162float(__float2bfloat16_rn(y[j]));  // the entry's bf16 values are what is quantised
    amax = fmaxf(amax, fabsf(y[j]));
  }
#pragma unroll
  for (int off = 1; off < kGroupThreads; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  float s;
  const uint8_t sc = fp4_scale_code(amax, &s);
  uint8_t* dst = a.kv_fp4_out + static_cast<int64_t>(b) * a.fp4_stride_b + i * kFp4Entry;
  uint32_t codes = 0u;
#pragma unroll
  for (int j = 0; j < CPT / 2; ++j) codes |= fp4_pair_code(y[2 * j], y[2 * j + 1], s) << (8 * j);
  if constexpr (CPT == 8)
    *reinterpret_cast<uint32_t*>(dst + 4 * t) = codes;
  else if constexpr (CPT == 4)
    *reinterpret_cast<uint16_t*>(dst + 2 * t) = static_cast<uint16_t>(codes);
  else
    dst[t] = static_cast<uint8_t>(codes);
  if (t % kGroupThreads == 0) dst[kDim / 2 + t * CPT / 16] = sc;
}

// The indexer's key entry ([hca_csa] "CSA：轻压缩 + 稀疏选择": its own
// compressor at head_dim 128, then a Hadamard rotation so that the keys
// quantise well to FP8), computed by one warp: the compressor's steps at
// width 128 with 4 channels per lane, then H_128/sqrt(128) as butterflies
// (two stages in registers, five across lanes), then E4M3 with
// round-to-nearest-even and saturation at +-448, stored at
// key_out[b*kv_stride_b + i*128].  Bulk mode: the e-th entry of the chunk;
// ring mode: the entry completing at q_pos[b], if any.  `red` is one float
// of shared memory for the warp.
template <int M>
__device__ __forceinline__ void index_key_entry(const CompressArgs& a, int b, int64_t e, int lane, float* red) {
  float y[4];
  int64_t i;
  const auto sync = [] { __syncwarp(); };
  if (!compress_values<M, 4, kIdxDim, decltype(sync), false, (M <= 4)>(a, b, e, lane, red, sync, y, &i)) return;
  // butterflies (a, b) -> (a + b, a - b) over channel distance 1, 2 (within
  // the lane's 4 channels), then 4 .. 64 (lanes 1 .. 16 apart)
  {
    const float s0 = y[0] + y[1], d0 = y[0] - y[1], s1 = y[2] + y[3], d1 = y[2] - y[3];
    y[0] = s0 + s1;
    y[1] = d0 + d1;
    y[2] = s0 - s1;
    y[3] = d0 - d1;
  }
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const bool upper = (lane >> st) & 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float o = __shfl_xor_sync(0xffffffffu, y[j], 1 << st);
      y[j] = upper ? o - y[j] : y[j] + o;
    }
  }
  constexpr float kInvSqrt128 = 0.088388347648318440550f;
  uint32_t codes = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    codes |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(y[j] * kInvSqrt128, __NV_SATFINITE, __NV_E4M3)) << (8 * j);
  *reinterpret_cast<uint32_t*>(a.key_out + static_cast<int64_t>(b) * a.kv_stride_b + i * kIdxDim + 4 * lane) = codes;
}

// The same key entry computed by 128 threads, one channel each (a latency
// form for one entry per sequence: the chain of dependent steps is a quarter
// of the one-warp form's).  t: 0..127, the thread's channel; red: 4 floats
// and xch: 128 floats of shared memory; sync(): a barrier over exactly the
// 128 threads.  The Hadamard butterflies run across lanes (channel distance
// 1..16) and through shared memory (32 and 64).
template <int M, class Sync>
__device__ __forceinline__ void index_key_entry_wide(const CompressArgs& a, int b, int t, float* red, float* xch,
                                                     Sync sync) {
  float y[1];
  int64_t i;
  if (!compress_values<M, 1, kIdxDim, Sync, false, (M <= 4)>(a, b, 0, t, red, sync, y, &i)) return;
  float v = y[0];
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const float o = __shfl_xor_sync(0xffffffffu, v, 1 << st);
    v = ((t >> st) & 1) ? o - v : v + o;
  }
#pragma unroll
  for (int st = 5; st < 7; ++st) {
    xch[t] = v;
    sync();
    const float o = xch[t ^ (1 << st)];
    sync();  // every thread has read its partner before the next stage writes
    v = ((t >> st) & 1) ? o - v : v + o;
  }
  constexpr float kInvSqrt128 = 0.088388347648318440550f;
  uint32_t code = static_cast<uint32_t>(__nv_cvt_float_to_fp8(v * kInvSqrt128, __NV_SATFINITE, __NV_E4M3));
  // four neighbouring channels' codes into one 32-bit store
  code |= __shfl_down_sync(0xffffffffu, code, 1) << 8;
  code |= __shfl_down_sync(0xffffffffu, code, 2) << 16;
  if ((t & 3) == 0)
    *reinterpret_cast<uint32_t*>(a.key_out + static_cast<int64_t>(b) * a.kv_stride_b + i * kIdxDim + t) = code;
}

// index_key_entry for the ratio a.m (1, 2, 4 or 8).
__device__ __forceinline__ void index_key_entry_m(const CompressArgs& a, int b, int64_t e, int lane, float* red) {
  switch (a.m) {
    case 1: index_key_entry<1>(a, b, e, lane, red); break;
    case 2: index_key_entry<2>(a, b, e, lane, red); break;
    case 4: index_key_entry<4>(a, b, e, lane, red); break;
    case 8: index_key_entry<8>(a, b, e, lane, red); break;
    default: break;
  }
}

// index_key_entry_wide for the ratio a.m (1, 2, 4 or 8).
template <class Sync>
__device__ __forceinline__ void index_key_entry_wide_m(const CompressArgs& a, int b, int t, float* red, float* xch,
                                                       Sync sync) {
  switch (a.m) {
    case 1: index_key_entry_wide<1>(a, b, t, red, xch, sync); break;
    case 2: index_key_entry_wide<2>(a, b, t, red, xch, sync); break;
    case 4: index_key_entry_wide<4>(a, b, t, red, xch, sync); break;
    case 8: index_key_entry_wide<8>(a, b, t, red, xch, sync); break;
    default: break;
  }
}

// The RoPE frequency table of the arguments (a->rope_turns from a->rope_theta).
void fill_rope(CompressArgs* a);

}  // namespace csa
