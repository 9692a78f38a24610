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
// be off by ~0.1 rad there.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace csa {
namespace {

constexpr int kThreads = kDim / 8;  // 64

__device__ __forceinline__ void load8(const uint16_t* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
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

  // Logits (Z + B) of the 2M slots, per channel.
  float la[M][8], lb[M][8];
  float mx[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mx[j] = -INFINITY;
#pragma unroll
  for (int r = 0; r < M; ++r) {
    float z[8], bias[8];
    load8(za[r] + d0, z);
    load8(a.Ba + r * D + d0, bias);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      la[r][j] = z[j] + bias[j];
      mx[j] = fmaxf(mx[j], la[r][j]);
    }
  }
#pragma unroll
  for (int r = 0; r < M; ++r) {
    if (has_prev) {
      float z[8], bias[8];
      load8(zb[r] + d0, z);
      load8(a.Bb + r * D + d0, bias);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        lb[r][j] = z[j] + bias[j];
        mx[j] = fmaxf(mx[j], lb[r][j]);
      }
    }
  }

  // Softmax-weighted sum of the C rows.
  constexpr float kLog2e = 1.4426950408889634f;
  float num[8], den[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) num[j] = den[j] = 0.f;
#pragma unroll
  for (int r = 0; r < M; ++r) {
    float c[8];
    load8(ca[r] + d0, c);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float w = exp2f((la[r][j] - mx[j]) * kLog2e);
      num[j] = fmaf(w, c[j], num[j]);
      den[j] += w;
    }
  }
  if (has_prev) {
#pragma unroll
    for (int r = 0; r < M; ++r) {
      float c[8];
      load8(cb[r] + d0, c);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = exp2f((lb[r][j] - mx[j]) * kLog2e);
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
  load8(a.rms_w + d0, w);
  float y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = x[j] * inv * w[j];

  // Partial RoPE on channels D-R .. D-1, interleaved pairs, position M*i.
  if (d0 >= D - kRope) {
    const double pos = static_cast<double>(M) * static_cast<double>(i);
    const double two_pi = 6.283185307179586476925286766559;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      const int jp = (d0 + 2 * pr - (D - kRope)) / 2;
      const double freq = pow(a.rope_theta, -2.0 * jp / static_cast<double>(kRope));
      double phi = pos * freq;
      phi -= two_pi * rint(phi / two_pi);
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

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t stream) {
  if (a.B <= 0) return cudaSuccess;
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
