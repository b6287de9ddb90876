// Decode: one query row per (slot, layer, head) attends non-causally over the
// valid encoder keys of the projection cache, out = softmax(scale * q.K^T) V
// ("Whisper: Trace One Encoder Tensor into Every Decoder Layer", "View 2 --
// expand one cross-attention operation": one query token, all key tokens,
// head_dim 64, scale 0.125).
//
// Split-T flash decoding with the lazy (online) softmax of SplitKV ("Caso de
// estudio: WhisperKit", §3): the keys of a row are cut into chunks of kChunk;
// each chunk is one CTA that
//   1. bulk-copies its K rows and V rows (contiguous in the head-major cache)
//      into shared memory with two cp.async.bulk copies,
//   2. computes the chunk's scores in fp32 (16 or 8 lanes per key row, warp
//      shuffle reduction), its max m and sum s of 2^(score - m),
//   3. accumulates sum_t 2^(score_t - m) V_t,
//   4. stores the partial (m, s, acc[64]) and counts itself done on the row's
//      arrival counter; the CTA that arrives last merges the row's partials
//      (M = max m_i, S = sum s_i 2^(m_i - M), out = sum acc_i 2^(m_i - M) / S),
//      writes out and resets the counter. No CTA ever waits for another.
// Scores are kept in base 2: q is pre-multiplied by scale * log2(e).
// Keys t >= key_len[b] are never copied and never enter the arithmetic; a row
// with no valid key gets out = 0.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace cxa {
namespace {

constexpr int kChunk = 64;          // keys per CTA
constexpr int kThreads = 128;       // 4 warps x 16 keys
constexpr int kPartFloats = 68;     // m, s, 2 pad, acc[64]
constexpr int kDh = 64;

template <bool kBF16>
struct RowTraits {
  static constexpr int kElemBytes = kBF16 ? 2 : 4;
  static constexpr int kRowBytes = kDh * kElemBytes;     // 256 / 128
  static constexpr int kLanesPerRow = kRowBytes / 16;    // 16 / 8
  static constexpr int kRowsPerPass = 32 / kLanesPerRow; // 2 / 4
  static constexpr int kElemsPerLane = 16 / kElemBytes;  // 4 / 8
};

// 16 bytes of a cache row -> fp32 values
template <bool kBF16>
__device__ __forceinline__ void unpack16(const uint4 u, float* f) {
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
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads)
    decode_split_kernel(const float* __restrict__ Q, const uint8_t* __restrict__ Kc,
                        const uint8_t* __restrict__ Vc, const int* __restrict__ key_len,
                        float* __restrict__ out, float* __restrict__ part,
                        unsigned int* __restrict__ counters, int T, int LH, int nchunk_max,
                        float qscale, unsigned int* status) {
  using R = RowTraits<kBF16>;
  constexpr int kRowsPerWarp = kChunk / (kThreads / 32);   // 16
  constexpr int kPasses = kRowsPerWarp / R::kRowsPerPass;  // 8 / 4

  __shared__ __align__(128) uint8_t sK[kChunk * R::kRowBytes];
  __shared__ __align__(128) uint8_t sV[kChunk * R::kRowBytes];
  __shared__ float s_score[kChunk];
  __shared__ float s_red[kThreads / 32][kDh];
  __shared__ __align__(8) uint64_t s_bar[2];
  __shared__ int s_last;

  const int chunk = blockIdx.x;
  const int lh = blockIdx.y;
  const int b = blockIdx.z;
  const int row = b * LH + lh;
  const int kl = min(max(__ldg(key_len + b), 0), T);
  const int t0 = chunk * kChunk;
  if (kl == 0) {
    if (chunk == 0 && threadIdx.x < kDh) out[static_cast<size_t>(row) * kDh + threadIdx.x] = 0.f;
    return;
  }
  if (t0 >= kl) return;
  const int n = min(kChunk, kl - t0);
  const int nch = (kl + kChunk - 1) / kChunk;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t barK = smem_u32(&s_bar[0]);
  const uint32_t barV = smem_u32(&s_bar[1]);

  if (threadIdx.x == 0) {
    mbar_init(barK, 1);
    mbar_init(barV, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const size_t off = (static_cast<size_t>(row) * T + t0) * R::kRowBytes;
    const uint32_t bytes = static_cast<uint32_t>(n) * R::kRowBytes;
    const uint64_t pol = policy_evict_first();
    mbar_arrive_expect_tx(barK, bytes);
    bulk_g2s_hint(smem_u32(sK), Kc + off, bytes, barK, pol);
    mbar_arrive_expect_tx(barV, bytes);
    bulk_g2s_hint(smem_u32(sV), Vc + off, bytes, barV, pol);
  }

  // this lane's slice of the query, pre-scaled into base-2 logits
  const int sub = lane % R::kLanesPerRow;
  const int rsub = lane / R::kLanesPerRow;
  float q[R::kElemsPerLane];
  {
    const float4* q4 = reinterpret_cast<const float4*>(Q + static_cast<size_t>(row) * kDh + sub * R::kElemsPerLane);
#pragma unroll
    for (int i = 0; i < R::kElemsPerLane / 4; ++i) {
      const float4 v = __ldg(q4 + i);
      q[4 * i + 0] = v.x * qscale;
      q[4 * i + 1] = v.y * qscale;
      q[4 * i + 2] = v.z * qscale;
      q[4 * i + 3] = v.w * qscale;
    }
  }

  bool ok = mbar_wait(barK, 0);
  // ---- scores
#pragma unroll
  for (int it = 0; it < kPasses; ++it) {
    const int r = warp * kRowsPerWarp + it * R::kRowsPerPass + rsub;
    float f[R::kElemsPerLane];
    unpack16<kBF16>(*reinterpret_cast<const uint4*>(sK + r * R::kRowBytes + sub * 16), f);
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < R::kElemsPerLane; ++e) dot = fmaf(q[e], f[e], dot);
#pragma unroll
    for (int off = R::kLanesPerRow / 2; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (sub == 0) s_score[r] = (r < n && ok) ? dot : -INFINITY;
  }
  __syncthreads();

  // ---- chunk max and sum (every warp computes them from shared memory)
  const float sa = s_score[lane];
  const float sb = s_score[lane + 32];
  float m = fmaxf(sa, sb);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float ssum = (lane < n ? exp2f(sa - m) : 0.f) + (lane + 32 < n ? exp2f(sb - m) : 0.f);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, off);

  // ---- weighted V rows
  ok = mbar_wait(barV, 0) && ok;
  float acc[R::kElemsPerLane];
#pragma unroll
  for (int e = 0; e < R::kElemsPerLane; ++e) acc[e] = 0.f;
#pragma unroll
  for (int it = 0; it < kPasses; ++it) {
    const int r = warp * kRowsPerWarp + it * R::kRowsPerPass + rsub;
    if (r < n && ok) {
      const float pr = exp2f(s_score[r] - m);
      float f[R::kElemsPerLane];
      unpack16<kBF16>(*reinterpret_cast<const uint4*>(sV + r * R::kRowBytes + sub * 16), f);
#pragma unroll
      for (int e = 0; e < R::kElemsPerLane; ++e) acc[e] = fmaf(pr, f[e], acc[e]);
    }
  }
#pragma unroll
  for (int off = R::kLanesPerRow; off < 32; off <<= 1)
#pragma unroll
    for (int e = 0; e < R::kElemsPerLane; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
  if (lane < R::kLanesPerRow) {
#pragma unroll
    for (int e = 0; e < R::kElemsPerLane; ++e) s_red[warp][sub * R::kElemsPerLane + e] = acc[e];
  }
  if (!ok && threadIdx.x == 0) atomicOr(status, 1u);
  __syncthreads();

  float* P = part + (static_cast<size_t>(row) * nchunk_max + chunk) * kPartFloats;
  if (threadIdx.x < kDh) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) a += s_red[w][threadIdx.x];
    P[4 + threadIdx.x] = a;
    if (threadIdx.x == 0) {
      P[0] = ok ? m : -INFINITY;
      P[1] = ok ? ssum : 0.f;
    }
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = atomicAdd(counters + row, 1u);
    s_last = (prev == static_cast<unsigned int>(nch - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA of this row: merge the partials
  __threadfence();
  if (threadIdx.x < kDh) {
    const float* P0 = part + static_cast<size_t>(row) * nchunk_max * kPartFloats;
    float M = -INFINITY;
    for (int i = 0; i < nch; ++i) M = fmaxf(M, __ldcg(P0 + i * kPartFloats));
    float S = 0.f, A = 0.f;
    for (int i = 0; i < nch; ++i) {
      const float mi = __ldcg(P0 + i * kPartFloats);
      const float w = mi == -INFINITY ? 0.f : exp2f(mi - M);
      S = fmaf(w, __ldcg(P0 + i * kPartFloats + 1), S);
      A = fmaf(w, __ldcg(P0 + i * kPartFloats + 4 + threadIdx.x), A);
    }
    out[static_cast<size_t>(row) * kDh + threadIdx.x] = S > 0.f ? A / S : 0.f;
  }
  if (threadIdx.x == 0) counters[row] = 0u;
}

size_t counters_bytes(int B, int L, int H) {
  const size_t n = static_cast<size_t>(B) * L * H * sizeof(unsigned int);
  return (n + 255) & ~static_cast<size_t>(255);
}

}  // namespace

size_t decode_workspace_bytes(int B, int T, int L, int H) {
  const size_t nchunk = static_cast<size_t>((T + kChunk - 1) / kChunk);
  return counters_bytes(B, L, H) + static_cast<size_t>(B) * L * H * nchunk * kPartFloats * sizeof(float);
}

size_t decode_counter_bytes(int B, int L, int H) { return counters_bytes(B, L, H); }

cudaError_t launch_decode(const DecodeLaunch& a, const DeviceInfo& dev, cudaStream_t stream,
                          std::string* msg) {
  (void)msg;
  const int LH = a.L * a.H;
  const int nchunk_max = (a.T + kChunk - 1) / kChunk;
  unsigned int* counters = static_cast<unsigned int*>(a.workspace);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + counters_bytes(a.B, a.L, a.H));
  const float qscale = a.scale * 1.4426950408889634f;   // scale * log2(e)
  dim3 grid(nchunk_max, LH, a.B);
  if (a.cache_bf16)
    decode_split_kernel<true><<<grid, kThreads, 0, stream>>>(
        a.Q, static_cast<const uint8_t*>(a.Kc), static_cast<const uint8_t*>(a.Vc), a.key_len, a.out, part,
        counters, a.T, LH, nchunk_max, qscale, dev.status_word);
  else
    decode_split_kernel<false><<<grid, kThreads, 0, stream>>>(
        a.Q, static_cast<const uint8_t*>(a.Kc), static_cast<const uint8_t*>(a.Vc), a.key_len, a.out, part,
        counters, a.T, LH, nchunk_max, qscale, dev.status_word);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace cxa
