// Cross-attention weights of selected (layer, head) pairs -- the alignment heads
// whose attention over encoder frames a decoder returns for word timestamps
// ("Caso de estudio: WhisperKit", §6: the cross-attention of specific alignment
// heads returns its weights, and their mean over heads is an extra output):
//
//   weights[b][k][t] = softmax_t(scale * q[b, l_k, h_k] . K[b, l_k, h_k, t])   t < key_len[b]
//                    = 0                                                    t >= key_len[b]
//   mean[b][t]       = (1 / nsel) sum_k weights[b][k][t]
//
// One CTA per (slot, selected head): its scores go to the weights row (one
// coalesced pass over the K rows, 16 lanes per fp32 row / 8 per bf16 row),
// then the row is normalised in place with a CTA-wide max and sum. A second
// kernel averages the selected heads.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <string>

#include "internal.h"

namespace cxa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float r = is_max ? -INFINITY : 0.f;
  for (int w = 0; w < kThreads / 32; ++w) r = is_max ? fmaxf(r, s_red[w]) : r + s_red[w];
  return r;
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads)
    alignment_weights_kernel(const float* __restrict__ Q, const uint8_t* __restrict__ Kc,
                             const int* __restrict__ key_len, const AlignHeads heads, float* __restrict__ weights,
                             int T, int L, int H, float qscale) {
  constexpr int kElem = kBF16 ? 2 : 4;
  constexpr int kRowBytes = 64 * kElem;
  constexpr int kLanesPerRow = kRowBytes / 16;          // 16 / 8
  constexpr int kEPL = 16 / kElem;                      // 4 / 8 channels per lane
  constexpr int kRowsPerIter = kThreads / kLanesPerRow; // 16 / 32 keys per CTA pass
  __shared__ float s_red[kThreads / 32];

  const int k = blockIdx.x, b = blockIdx.y;
  const int l = heads.l[k], h = heads.h[k];
  const int n = min(max(__ldg(key_len + b), 0), T);
  const long long crow = (static_cast<long long>(b) * L + l) * H + h;
  float* wrow = weights + (static_cast<long long>(b) * gridDim.x + k) * T;
  const int sub = threadIdx.x % kLanesPerRow, r0 = threadIdx.x / kLanesPerRow;

  float q[kEPL];
#pragma unroll
  for (int e4 = 0; e4 < kEPL / 4; ++e4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(Q + crow * 64 + sub * kEPL) + e4);
    q[4 * e4 + 0] = v.x * qscale;
    q[4 * e4 + 1] = v.y * qscale;
    q[4 * e4 + 2] = v.z * qscale;
    q[4 * e4 + 3] = v.w * qscale;
  }
  // scores (base 2) into the output row, running max per thread
  float mx = -INFINITY;
  for (int t0 = 0; t0 < n; t0 += kRowsPerIter) {   // the same trip count for every lane (shuffles below)
    const int t = t0 + r0;
    const bool valid = t < n;
    const uint4 u = valid ? __ldg(reinterpret_cast<const uint4*>(Kc + (crow * T + t) * kRowBytes) + sub)
                          : make_uint4(0u, 0u, 0u, 0u);
    float f[kEPL];
    if constexpr (kBF16) {
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
      f[0] = __uint_as_float(u.x);
      f[1] = __uint_as_float(u.y);
      f[2] = __uint_as_float(u.z);
      f[3] = __uint_as_float(u.w);
    }
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < kEPL; ++e) dot = fmaf(q[e], f[e], dot);
#pragma unroll
    for (int off = kLanesPerRow / 2; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (valid) {
      if (sub == 0) wrow[t] = dot;
      mx = fmaxf(mx, dot);
    }
  }
  const float M = block_reduce(mx, true, s_red);        // the CTA's writes of wrow are visible after its barriers
  float sum = 0.f;
  for (int t = threadIdx.x; t < n; t += kThreads) {
    const float p = exp2f(wrow[t] - M);
    wrow[t] = p;
    sum += p;
  }
  const float S = block_reduce(sum, false, s_red);
  const float inv = S > 0.f ? 1.f / S : 0.f;
  for (int t = threadIdx.x; t < T; t += kThreads) wrow[t] = t < n ? wrow[t] * inv : 0.f;
}

__global__ void __launch_bounds__(kThreads)
    head_mean_kernel(const float* __restrict__ weights, float* __restrict__ mean, int nsel, int T) {
  const int b = blockIdx.y;
  const int t = blockIdx.x * kThreads + threadIdx.x;
  if (t >= T) return;
  float s = 0.f;
  for (int k = 0; k < nsel; ++k) s += weights[(static_cast<long long>(b) * nsel + k) * T + t];
  mean[static_cast<long long>(b) * T + t] = s / static_cast<float>(nsel);
}

}  // namespace

cudaError_t launch_alignment(const AlignLaunch& a, cudaStream_t stream) {
  const dim3 grid(a.heads.n, a.B);
  const float qscale = a.scale * 1.4426950408889634f;
  if (a.cache_bf16)
    alignment_weights_kernel<true><<<grid, kThreads, 0, stream>>>(a.Q, static_cast<const uint8_t*>(a.Kc), a.key_len,
                                                                  a.heads, a.weights, a.T, a.L, a.H, qscale);
  else
    alignment_weights_kernel<false><<<grid, kThreads, 0, stream>>>(a.Q, static_cast<const uint8_t*>(a.Kc), a.key_len,
                                                                   a.heads, a.weights, a.T, a.L, a.H, qscale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launches(1);
  if (a.mean != nullptr) {
    head_mean_kernel<<<dim3((a.T + kThreads - 1) / kThreads, a.B), kThreads, 0, stream>>>(a.weights, a.mean,
                                                                                          a.heads.n, a.T);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
  }
  return cudaSuccess;
}

}  // namespace cxa
