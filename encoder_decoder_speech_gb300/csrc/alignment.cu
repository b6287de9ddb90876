// Cross-attention weights of selected (layer, head) pairs -- the alignment heads
// whose attention over encoder frames a decoder returns for word timestamps
// ("Caso de estudio: WhisperKit", §6: the cross-attention of specific alignment
// heads returns its weights, and their mean over heads is an extra output):
//
//   weights[b][k][t] = softmax_t(scale * q[b, l_k, h_k] . K[b, l_k, h_k, t])   t < key_len[b]
//                    = 0                                                    t >= key_len[b]
//   mean[b][t]       = (1 / nsel) sum_k weights[b][k][t]
//
// Three launches, chained by programmatic dependent launch:
//  1. scores: a CTA per (block of 128 keys, selected head, slot) writes the base-2
//     logits scale * log2(e) * q . K_t into the weights row, every thread's row
//     loads of the block issued together (16 lanes per fp32 row / 8 per bf16 row);
//  2. normalise: a CTA per (selected head, slot) takes the row max, sums 2^(s - max)
//     and scales the row, writing 0 past key_len;
//  3. mean over the selected heads (optional).
// The K rows of the selected heads are the only large reads; splitting each row
// over many CTAs keeps enough of them in flight.
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

constexpr int kBlockKeys = 128;   // keys per score CTA

template <bool kBF16>
__global__ void __launch_bounds__(kThreads)
    alignment_scores_kernel(const float* __restrict__ Q, const uint8_t* __restrict__ Kc,
                            const int* __restrict__ key_len, const AlignHeads heads, float* __restrict__ weights,
                            int T, int L, int H, float qscale) {
  constexpr int kElem = kBF16 ? 2 : 4;
  constexpr int kRowBytes = 64 * kElem;
  constexpr int kLanesPerRow = kRowBytes / 16;          // 16 / 8
  constexpr int kEPL = 16 / kElem;                      // 4 / 8 channels per lane
  constexpr int kRowsPerPass = kThreads / kLanesPerRow; // 16 / 32 keys per CTA pass
  constexpr int kPasses = kBlockKeys / kRowsPerPass;    // 8 / 4
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int k = blockIdx.y, b = blockIdx.z;
  const int n = min(max(__ldg(key_len + b), 0), T);
  const int t0 = blockIdx.x * kBlockKeys;
  if (t0 >= n) return;
  const int l = heads.l[k], h = heads.h[k];
  const long long crow = (static_cast<long long>(b) * L + l) * H + h;
  float* wrow = weights + (static_cast<long long>(b) * gridDim.y + k) * T;
  const int sub = threadIdx.x % kLanesPerRow, r0 = threadIdx.x / kLanesPerRow;
  // the cache rows first (no decode writes them), then Q and the weights (which
  // neighbouring kernels may produce or read)
  uint4 u[kPasses];
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int t = t0 + ps * kRowsPerPass + r0;
    u[ps] = t < n ? __ldg(reinterpret_cast<const uint4*>(Kc + (crow * T + t) * kRowBytes) + sub)
                  : make_uint4(0u, 0u, 0u, 0u);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float q[kEPL];
#pragma unroll
  for (int e4 = 0; e4 < kEPL / 4; ++e4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(Q + crow * 64 + sub * kEPL) + e4);
    q[4 * e4 + 0] = v.x * qscale;
    q[4 * e4 + 1] = v.y * qscale;
    q[4 * e4 + 2] = v.z * qscale;
    q[4 * e4 + 3] = v.w * qscale;
  }
  float dot[kPasses];
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    float f[kEPL];
    if constexpr (kBF16) {
      const uint32_t w[4] = {u[ps].x, u[ps].y, u[ps].z, u[ps].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
      f[0] = __uint_as_float(u[ps].x);
      f[1] = __uint_as_float(u[ps].y);
      f[2] = __uint_as_float(u[ps].z);
      f[3] = __uint_as_float(u[ps].w);
    }
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < kEPL; ++e) d = fmaf(q[e], f[e], d);
    dot[ps] = d;
  }
#pragma unroll
  for (int off = kLanesPerRow / 2; off >= 1; off >>= 1)
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) dot[ps] += __shfl_xor_sync(0xffffffffu, dot[ps], off);
  if (sub == 0) {
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
      const int t = t0 + ps * kRowsPerPass + r0;
      if (t < n) wrow[t] = dot[ps];
    }
  }
}

// Row (slot blockIdx.y, selected head blockIdx.x) of base-2 logits -> softmax weights.
__global__ void __launch_bounds__(kThreads)
    alignment_normalise_kernel(const int* __restrict__ key_len, float* __restrict__ weights, int T) {
  __shared__ float s_red[kThreads / 32];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.y;
  const int n = min(max(__ldg(key_len + b), 0), T);
  float* wrow = weights + (static_cast<long long>(b) * gridDim.x + blockIdx.x) * T;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the scores
  float mx = -INFINITY;
  for (int t = threadIdx.x; t < n; t += kThreads) mx = fmaxf(mx, wrow[t]);
  const float M = block_reduce(mx, true, s_red);
  float sum = 0.f;
  for (int t = threadIdx.x; t < n; t += kThreads) sum += exp2f(wrow[t] - M);
  const float S = block_reduce(sum, false, s_red);
  const float inv = S > 0.f ? 1.f / S : 0.f;
  for (int t = threadIdx.x; t < T; t += kThreads) wrow[t] = t < n ? exp2f(wrow[t] - M) * inv : 0.f;
}

__global__ void __launch_bounds__(kThreads)
    head_mean_kernel(const float* __restrict__ weights, float* __restrict__ mean, int nsel, int T) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.y;
  const int t = blockIdx.x * kThreads + threadIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the normalised weights
  if (t >= T) return;
  float s = 0.f;
  for (int k = 0; k < nsel; ++k) s += weights[(static_cast<long long>(b) * nsel + k) * T + t];
  mean[static_cast<long long>(b) * T + t] = s / static_cast<float>(nsel);
}

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace

cudaError_t launch_alignment(const AlignLaunch& a, cudaStream_t stream) {
  const float qscale = a.scale * 1.4426950408889634f;
  const dim3 grid((a.T + kBlockKeys - 1) / kBlockKeys, a.heads.n, a.B);
  const uint8_t* Kc = static_cast<const uint8_t*>(a.Kc);
  cudaError_t e = a.cache_bf16
                      ? launch_pdl(alignment_scores_kernel<true>, grid, stream, a.Q, Kc, a.key_len, a.heads,
                                   a.weights, a.T, a.L, a.H, qscale)
                      : launch_pdl(alignment_scores_kernel<false>, grid, stream, a.Q, Kc, a.key_len, a.heads,
                                   a.weights, a.T, a.L, a.H, qscale);
  if (e != cudaSuccess) return e;
  e = launch_pdl(alignment_normalise_kernel, dim3(a.heads.n, a.B), stream, a.key_len, a.weights, a.T);
  if (e != cudaSuccess) return e;
  if (a.mean != nullptr)
    e = launch_pdl(head_mean_kernel, dim3((a.T + kThreads - 1) / kThreads, a.B), stream,
                   static_cast<const float*>(a.weights), a.mean, a.heads.n, a.T);
  return e;
}

}  // namespace cxa
