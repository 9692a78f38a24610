// Overlapped CSA compressor: per-channel softmax pooling over 2m slots,
// RMSNorm, partial RoPE.  Page "CSA / HCA" (zdszero, hca_csa), section
// "CSA 的重叠窗口" (Softmax_row and C_i^Comp equations, i = 0 boundary);
// RoPE position = first token of the entry's block ("DeepSeek-V4 CSA/HCA 与
// DeepSeek-V4.1 CSA2" §7.4); decode emission only at a block boundary
// ("DeepSeek-V4 的 KV 压缩：从删 token 误解到预算检索" §9.3).
//
// Streaming kernel: one 64-thread CTA per (entry, sequence); thread t owns
// channels 8t..8t+7 and reads each of the 4*m source rows it needs with one
// 16-byte load (a warp reads 512 contiguous bytes of a row).  Softmax,
// normalisation and rotation are fp32; the RoPE angle is formed and reduced
// modulo 2*pi in fp64 because positions reach 2^20 and an fp32 angle would
// be off by ~0.1 rad there.  The 32 inverse frequencies are computed once on
// the host (fp64) and passed with the arguments, so the device does one
// multiply, one reduction and one fp32 sincos per channel pair.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kThreads = kDim / 8;  // 64

__device__ __forceinline__ void unpack8(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void store8(uint16_t* p, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <int M>
__global__ void __launch_bounds__(kThreads) compress_kernel(const CompressArgs a) {
  const int b = blockIdx.y;
  const int d0 = threadIdx.x * 8;
  constexpr int D = kDim;

  // Locate entry i and the rows of block i (a stream) and block i-1 (b stream).
  int64_t i;
  const uint16_t *ca[M], *za[M], *cb[M], *zb[M];
  bool has_prev;
  if (a.mode == 0) {
    const int64_t e = blockIdx.x;
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
    const int64_t t = a.q_pos[b];
    if (t < 0 || (t + 1) % M != 0) return;  // no block completes at this step
    i = (t + 1) / M - 1;
    if (i >= a.n_cap) {
      if (threadIdx.x == 0) record_error(a.status, kErrIndexRange);
      return;
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

  // Issue every load of the entry first (one memory round trip), then math.
  uint4 zr[2 * M], cr[2 * M], br[2 * M];
#pragma unroll
  for (int r = 0; r < M; ++r) {
    zr[r] = __ldg(reinterpret_cast<const uint4*>(za[r] + d0));
    cr[r] = __ldg(reinterpret_cast<const uint4*>(ca[r] + d0));
    br[r] = __ldg(reinterpret_cast<const uint4*>(a.Ba + r * D + d0));
    if (has_prev) {
      zr[M + r] = __ldg(reinterpret_cast<const uint4*>(zb[r] + d0));
      cr[M + r] = __ldg(reinterpret_cast<const uint4*>(cb[r] + d0));
      br[M + r] = __ldg(reinterpret_cast<const uint4*>(a.Bb + r * D + d0));
    }
  }
  const uint4 wr = __ldg(reinterpret_cast<const uint4*>(a.rms_w + d0));
  const int slots = has_prev ? 2 * M : M;  // block i-1 slots are absent for entry 0

  // Logits (Z + B) of the slots, per channel, and their maximum.
  float lg[2 * M][8];
  float mx[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mx[j] = -INFINITY;
#pragma unroll
  for (int r = 0; r < 2 * M; ++r) {
    if (r < slots) {
      float z[8], bias[8];
      unpack8(zr[r], z);
      unpack8(br[r], bias);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        lg[r][j] = z[j] + bias[j];
        mx[j] = fmaxf(mx[j], lg[r][j]);
      }
    }
  }

  // Softmax-weighted sum of the C rows.
  constexpr float kLog2e = 1.4426950408889634f;
  float num[8], den[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) num[j] = den[j] = 0.f;
#pragma unroll
  for (int r = 0; r < 2 * M; ++r) {
    if (r < slots) {
      float c[8];
      unpack8(cr[r], c);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = exp2f((lg[r][j] - mx[j]) * kLog2e);
        num[j] = fmaf(w, c[j], num[j]);
        den[j] += w;
      }
    }
  }
  float x[8];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    x[j] = num[j] / den[j];
    ss = fmaf(x[j], x[j], ss);
  }

  // RMSNorm over the 512 channels: warp sums, then the two warps combine.
  __shared__ float warp_ss[kThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
  __syncthreads();
  const float total = warp_ss[0] + warp_ss[1];
  const float inv = rsqrtf(total / static_cast<float>(D) + a.rms_eps);
  float w[8];
  unpack8(wr, w);
  float y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = x[j] * inv * w[j];

  // Partial RoPE on channels D-R .. D-1, interleaved pairs, position M*i.
  if (d0 >= D - kRope) {
    const double pos = static_cast<double>(M) * static_cast<double>(i);
    const double two_pi = 6.283185307179586476925286766559;
    const double inv_two_pi = 0.15915494309189533576888376337251;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      const int jp = (d0 + 2 * pr - (D - kRope)) / 2;
      double phi = pos * a.inv_freq[jp];
      phi = fma(-two_pi, rint(phi * inv_two_pi), phi);
      float s, c;
      sincosf(static_cast<float>(phi), &s, &c);
      const float u = y[2 * pr], v = y[2 * pr + 1];
      y[2 * pr] = u * c - v * s;
      y[2 * pr + 1] = u * s + v * c;
    }
  }

  store8(a.kv_out + static_cast<int64_t>(b) * a.kv_stride_b + i * D + d0, y);
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& args, cudaStream_t stream) {
  if (args.B <= 0) return cudaSuccess;
  CompressArgs a = args;
  for (int j = 0; j < kRope / 2; ++j) a.inv_freq[j] = pow(a.rope_theta, -2.0 * j / static_cast<double>(kRope));
  dim3 grid(a.mode == 0 ? static_cast<unsigned>(a.n_new) : 1u, static_cast<unsigned>(a.B));
  if (grid.x == 0) return cudaSuccess;
  switch (a.m) {
    case 1: compress_kernel<1><<<grid, kThreads, 0, stream>>>(a); break;
    case 2: compress_kernel<2><<<grid, kThreads, 0, stream>>>(a); break;
    case 4: compress_kernel<4><<<grid, kThreads, 0, stream>>>(a); break;
    case 8: compress_kernel<8><<<grid, kThreads, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return counted(cudaGetLastError());
}

}  // namespace csa
