// Cross-attention weights of selected (layer, head) pairs -- the alignment heads
// whose attention over encoder frames a decoder returns for word timestamps
// ("Caso de estudio: WhisperKit", §6: the cross-attention of specific alignment
// heads returns its weights, and their mean over heads is an extra output):
//
//   weights[b][k][t] = softmax_t(scale * q[b, l_k, h_k] . K[b, l_k, h_k, t])   t < key_len[b]
//                    = 0                                                    t >= key_len[b]
//   mean[b][t]       = (1 / nsel) sum_k weights[b][k][t]
//
// One launch. Slot b is a cluster of C CTAs (the largest of 16, 8, 4, 2, 1 whose
// B clusters are resident together); CTA x takes the keys [x*tc, (x+1)*tc) of the
// slot's valid range for EVERY selected head, so the head mean of a key needs
// nothing from other CTAs. The only cross-CTA step is the softmax denominator:
//  1. scores: each head's key range is one contiguous span of the cache; the CTA
//     streams its spans in 6 KB bulk copies through a 16-stage shared-memory ring.
//     Chunk j belongs to warp j % 8 alone, which waits for it, takes the dot
//     products of its rows (16 lanes per fp32 row / 8 per bf16 row, the 8 rows'
//     reductions interleaved) and refills the stage with chunk j + 16; the first
//     copies are issued before the grid dependency wait. The base-2 logits
//     scale*log2(e)*q.K_t are staged in shared memory (or, when nsel times the
//     CTA's keys exceeds 2048, in the weights rows);
//  2. per head, a group of lanes takes the max and the sum of 2^(logit - max)
//     over the CTA's keys and stores the pair into every cluster CTA's shared
//     memory (distributed shared memory);
//  3. after one cluster barrier each CTA merges the C pairs of every head from
//     its own shared memory (log-sum-exp);
//  4. every CTA writes the weights of its own keys and their mean over heads,
//     and zeroes its share of the keys t >= key_len[b].
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>

#include "cluster.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace cxa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// The K ring: kStages chunks of kChunkBytes. Two shapes, chosen per launch (timed on
// GB300): 16 x 6 KB (two CTAs per SM) and 8 x 8 KB (three per SM, so that a slot's
// cluster can be twice as large when the wide ring limits it).
template <int kChunkB, int kStg>
struct Ring {
  static constexpr int kChunkBytes = kChunkB;
  static constexpr int kStages = kStg;                            // warp w owns stages w, w + 8, ...
  static constexpr size_t kBytes = static_cast<size_t>(kStg) * kChunkB;
  static_assert(kStg % 8 == 0 && kChunkB % 1024 == 0, "ring shape");
};
using RingWide = Ring<6144, 16>;
using RingNarrow = Ring<8192, 8>;

template <bool kBF16, int kChunkB>
struct RowGeom {
  static constexpr int kElem = kBF16 ? 2 : 4;
  static constexpr int kRowBytes = 64 * kElem;
  static constexpr int kLanesPerRow = kRowBytes / 16;           // 16 / 8
  static constexpr int kEPL = 16 / kElem;                       // 4 / 8 channels per lane
  static constexpr int kRowsPerWarpPass = 32 / kLanesPerRow;    // 2 / 4
  static constexpr int kChunkBytes = kChunkB;
  static constexpr int kChunkKeys = kChunkBytes / kRowBytes;    // 24 / 48
  static constexpr int kWarpPasses = kChunkKeys / kRowsPerWarpPass;   // 12: one interleaved reduction
};
constexpr int kStageFloats = 2048;   // logits held in shared memory when nsel * keys per CTA fits
constexpr int kMaxCluster = 16;

// Dynamic shared memory: the ring, the logits, the scaled queries [nsel][64] and the
// partials [nsel][C] (max, then sum) every cluster CTA stores into every other.
template <class RG>
__host__ __device__ constexpr size_t dyn_smem_bytes(int nsel, int C) {
  return RG::kBytes + kStageFloats * sizeof(float) + static_cast<size_t>(nsel) * 64 * sizeof(float) +
         static_cast<size_t>(nsel) * C * 2 * sizeof(float);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <bool kBF16>
__device__ __forceinline__ void unpack(const uint4 u, float (&f)[16 / (kBF16 ? 2 : 4)]) {
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

template <bool kBF16, class RG>
__global__ void __launch_bounds__(kThreads)
    alignment_kernel(const float* __restrict__ Q, const uint8_t* __restrict__ Kc, const int* __restrict__ key_len,
                     const AlignHeads heads, float* weights, float* __restrict__ mean, int T, int L, int H,
                     float qscale, unsigned int* status) {
  using G = RowGeom<kBF16, RG::kChunkBytes>;
  constexpr int kStages = RG::kStages;
  constexpr size_t kRingBytes = RG::kBytes;
  extern __shared__ __align__(128) uint8_t ring[];              // see dyn_smem_bytes
  __shared__ float s_M[kMaxAlignHeads], s_inv[kMaxAlignHeads];  // merged max and 1 / sum
  __shared__ __align__(8) uint64_t bars[kStages];               // full[s]: chunk landed
  __shared__ int s_last[kStages];                               // last chunk issued into stage s
  __shared__ int s_abort;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  cluster_arrive();   // this CTA is running; peers wait for that before storing into its shared memory
  const int C = gridDim.x, x = blockIdx.x, b = blockIdx.y, nsel = heads.n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(smem_u32(&bars[st]), 1);
      s_last[st] = -1;
    }
    s_abort = 0;
    fence_mbar_init();
  }
  const int n = min(max(__ldg(key_len + b), 0), T);
  const int tc = (n + C - 1) / C;
  const int t_lo = min(n, x * tc);
  const int cnt = min(n, t_lo + tc) - t_lo;
  const int nchk = (cnt + G::kChunkKeys - 1) / G::kChunkKeys;   // chunks per head
  const int nchunks = nsel * nchk;                              // chunk j: head j / nchk, part j % nchk
  float* wslot = weights + static_cast<long long>(b) * nsel * T;
  volatile int* abort_flag = &s_abort;
  // the CTA's logits: [nsel][cnt] in shared memory when they fit, else in place in
  // the weights rows (same code through a generic pointer)
  const bool lg_smem = nsel * cnt <= kStageFloats;
  float* const s_lg = reinterpret_cast<float*>(ring + kRingBytes);
  float* const s_q = s_lg + kStageFloats;                       // [nsel][64]
  float* const s_pm = s_q + nsel * 64;                          // [nsel][C] partial max of CTA r at [k][r]
  float* const s_ps = s_pm + nsel * C;                          // [nsel][C] partial sum
  float* stage = lg_smem ? s_lg : wslot + t_lo;
  const long long ldst = lg_smem ? cnt : T;

  auto issue = [&](int j) {
    const int st = j % kStages, k = j / nchk, c = j - k * nchk;
    const int rows = min(G::kChunkKeys, cnt - c * G::kChunkKeys);
    const long long crow = (static_cast<long long>(b) * L + heads.l[k]) * H + heads.h[k];
    const uint32_t full = smem_u32(&bars[st]);
    const uint32_t bytes = static_cast<uint32_t>(rows) * G::kRowBytes;
    s_last[st] = j;
    mbar_arrive_expect_tx(full, bytes);
    bulk_g2s(smem_u32(ring + st * G::kChunkBytes), Kc + (crow * T + t_lo + c * G::kChunkKeys) * G::kRowBytes,
             bytes, full);
  };
  __syncthreads();                                              // the barriers are initialised
  // the cache rows and key_len first (no decode writes them); Q and the weights
  // after the wait (neighbouring kernels may produce or read them). Chunk j is
  // processed by warp j % 8, which also refills its stage with chunk j + kStages.
  if (lane == 0)
    for (int j = warp; j < min(nchunks, kStages); j += kWarps) issue(j);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = tid; i < nsel * 16; i += kThreads) {
    const int k = i >> 4, c4 = i & 15;
    const long long crow = (static_cast<long long>(b) * L + heads.l[k]) * H + heads.h[k];
    float4 v = __ldg(reinterpret_cast<const float4*>(Q + crow * 64) + c4);
    v.x *= qscale;
    v.y *= qscale;
    v.z *= qscale;
    v.w *= qscale;
    reinterpret_cast<float4*>(s_q)[i] = v;
  }
  __syncthreads();

  // ---- 1. scores of every chunk, staged as base-2 logits
  const int sub = lane % G::kLanesPerRow, grp = lane / G::kLanesPerRow;
  bool ok = true;
  for (int j = warp; j < nchunks; j += kWarps) {
    const int st = j % kStages, k = j / nchk, c = j - k * nchk;
    if (ok && !mbar_wait(smem_u32(&bars[st]), static_cast<uint32_t>((j / kStages) & 1), abort_flag)) {
      ok = false;
      *abort_flag = 1;
      atomicOr(status, 1u);
    }
    const int rows = ok ? min(G::kChunkKeys, cnt - c * G::kChunkKeys) : 0;
    const uint8_t* tile = ring + st * G::kChunkBytes + sub * 16;
    float q[G::kEPL];
#pragma unroll
    for (int e4 = 0; e4 < G::kEPL / 4; ++e4) {
      const float4 v = reinterpret_cast<const float4*>(s_q + k * 64 + sub * G::kEPL)[e4];
      q[4 * e4 + 0] = v.x;
      q[4 * e4 + 1] = v.y;
      q[4 * e4 + 2] = v.z;
      q[4 * e4 + 3] = v.w;
    }
    float* lg = stage + k * ldst + c * G::kChunkKeys;
    float dot[G::kWarpPasses];
#pragma unroll
    for (int i = 0; i < G::kWarpPasses; ++i) {
      const int r = i * G::kRowsPerWarpPass + grp;
      const uint4 u = r < rows ? *reinterpret_cast<const uint4*>(tile + r * G::kRowBytes) : make_uint4(0u, 0u, 0u, 0u);
      float f[G::kEPL];
      unpack<kBF16>(u, f);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < G::kEPL; ++e) d = fmaf(q[e], f[e], d);
      dot[i] = d;
    }
#pragma unroll
    for (int off = G::kLanesPerRow / 2; off >= 1; off >>= 1)
#pragma unroll
      for (int i = 0; i < G::kWarpPasses; ++i) dot[i] += __shfl_xor_sync(0xffffffffu, dot[i], off);
    if (sub == 0) {
#pragma unroll
      for (int i = 0; i < G::kWarpPasses; ++i) {
        const int r = i * G::kRowsPerWarpPass + grp;
        if (r < rows) lg[r] = dot[i];
      }
    }
    __syncwarp();
    if (lane == 0 && j + kStages < nchunks && *abort_flag == 0) issue(j + kStages);
  }
  __syncthreads();
  if (*abort_flag != 0 && tid == 0) {
    // let the copies still in flight land before the shared memory is released
    for (int st = 0; st < kStages; ++st)
      if (s_last[st] >= 0) mbar_wait(smem_u32(&bars[st]), static_cast<uint32_t>((s_last[st] / kStages) & 1));
  }

  // ---- 2. per-head partial max and sum over this CTA's keys, by groups of gl lanes
  //         (a warp per head up to 8 heads, fewer lanes per head beyond), stored into
  //         every cluster CTA's partial arrays (every peer has started: see the
  //         arrive at the top)
  cluster_wait();
  {
    const int gl = nsel <= 8 ? 32 : nsel <= 16 ? 16 : nsel <= 32 ? 8 : 4;
    const int gi = tid / gl, gsub = tid % gl, ngroups = kThreads / gl;
    for (int k0 = 0; k0 < nsel; k0 += ngroups) {              // uniform trip count: shuffles stay converged
      const int k = k0 + gi;
      const float* lk = stage + min(k, nsel - 1) * ldst;
      float m = -INFINITY;
      if (k < nsel)
        for (int t = gsub; t < cnt; t += gl) m = fmaxf(m, lk[t]);
      for (int off = gl / 2; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float s = 0.f;
      if (k < nsel)
        for (int t = gsub; t < cnt; t += gl) s += exp2f(lk[t] - m);
      for (int off = gl / 2; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (k < nsel)
        for (int r = gsub; r < C; r += gl) {                    // lanes r, r + gl, ... store into CTA r
          st_dsmem(s_pm + k * C + x, static_cast<uint32_t>(r), m);
          st_dsmem(s_ps + k * C + x, static_cast<uint32_t>(r), s);
        }
    }
  }
  cluster_sync();     // every partial has arrived; nothing remote is touched after this

  // ---- 3. merge each head's C partials (log-sum-exp)
  for (int k = warp; k < nsel; k += kWarps) {
    const float m = lane < C ? s_pm[k * C + lane] : -INFINITY;
    const float s = lane < C ? s_ps[k * C + lane] : 0.f;
    const float M = warp_max(m);
    const float S = warp_sum(s > 0.f ? s * exp2f(m - M) : 0.f);
    if (lane == 0) {
      s_M[k] = M;
      s_inv[k] = S > 0.f ? 1.f / S : 0.f;
    }
  }
  __syncthreads();

  // ---- 4. normalise this CTA's keys, their head mean, and its share of the padding
  const float inv_nsel = 1.f / static_cast<float>(nsel);
  float* mrow = mean != nullptr ? mean + static_cast<long long>(b) * T : nullptr;
  for (int t = t_lo + tid; t < t_lo + cnt; t += kThreads) {
    float acc = 0.f;
    for (int k = 0; k < nsel; ++k) {
      const float w = exp2f(stage[k * ldst + (t - t_lo)] - s_M[k]) * s_inv[k];
      wslot[static_cast<long long>(k) * T + t] = w;
      acc += w;
    }
    if (mrow != nullptr) mrow[t] = acc * inv_nsel;
  }
  const int zc = (T - n + C - 1) / C;
  const int z_lo = min(T, n + x * zc), z_hi = min(T, z_lo + zc);
  for (int t = z_lo + tid; t < z_hi; t += kThreads) {
    for (int k = 0; k < nsel; ++k) wslot[static_cast<long long>(k) * T + t] = 0.f;
    if (mrow != nullptr) mrow[t] = 0.f;
  }
}

// Largest cluster size C in {16, 8, 4, 2, 1} whose B clusters are all resident at
// once (one wave; 16 needs the non-portable size), else 1. The resident-cluster
// counts depend on the shared memory of the launch (nsel) and are queried once per
// device and head count.
template <bool kBF16, class RG>
int cluster_size(int B, int nsel, const DeviceInfo& dev) {
  static std::mutex mu;
  static int fit[128][kMaxAlignHeads + 1][5] = {};  // resident clusters of size 16, 8, 4, 2, 1
  static bool attr[128] = {}, big[128] = {}, queried[128][kMaxAlignHeads + 1] = {};
  const int dv = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!attr[dv]) {
    if (cudaFuncSetAttribute(alignment_kernel<kBF16, RG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(dyn_smem_bytes<RG>(kMaxAlignHeads, kMaxCluster))) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    big[dv] = cudaFuncSetAttribute(alignment_kernel<kBF16, RG>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
              cudaSuccess;
    cudaGetLastError();
    attr[dv] = true;
  }
  if (!queried[dv][nsel]) {
    for (int i = 0; i < 5; ++i) {
      const int c = 16 >> i;
      int n = 0;
      if (c <= 8 || big[dv]) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = dyn_smem_bytes<RG>(nsel, c);
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = c;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, alignment_kernel<kBF16, RG>, &cfg) != cudaSuccess) n = 0;
      }
      fit[dv][nsel][i] = n;
    }
    cudaGetLastError();
    queried[dv][nsel] = true;
  }
  for (int i = 0; i < 5; ++i)
    if (fit[dv][nsel][i] >= B) return 16 >> i;
  return 1;
}

template <bool kBF16, class RG>
cudaError_t launch_ring(const AlignLaunch& a, const DeviceInfo& dev, cudaStream_t stream, int C) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.B, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn_smem_bytes<RG>(a.heads.n, C);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const float qscale = a.scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&cfg, alignment_kernel<kBF16, RG>, a.Q, static_cast<const uint8_t*>(a.Kc), a.key_len,
                            a.heads, a.weights, a.mean, a.T, a.L, a.H, qscale, dev.status_word);
}

// The wide ring, unless the narrow one lets a slot's cluster be larger.
template <bool kBF16>
cudaError_t launch(const AlignLaunch& a, const DeviceInfo& dev, cudaStream_t stream) {
  const int Cw = cluster_size<kBF16, RingWide>(a.B, a.heads.n, dev);
  if (Cw < 0) return cudaErrorInvalidValue;
  if (Cw < kMaxCluster) {
    const int Cn = cluster_size<kBF16, RingNarrow>(a.B, a.heads.n, dev);
    if (Cn > Cw) return launch_ring<kBF16, RingNarrow>(a, dev, stream, Cn);
  }
  return launch_ring<kBF16, RingWide>(a, dev, stream, Cw);
}

}  // namespace

cudaError_t launch_alignment(const AlignLaunch& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (a.B > 65535) return cudaErrorInvalidValue;
  const cudaError_t e = a.cache_bf16 ? launch<true>(a, dev, stream) : launch<false>(a, dev, stream);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace cxa
