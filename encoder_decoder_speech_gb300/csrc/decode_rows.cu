// Decode for short streams: the latency shape of the one-query decode step.
//
// Same operation as the persistent stream kernel (decode.cu): one query row per
// (slot, layer, head) attends non-causally over the valid encoder keys, out =
// softmax(scale * q.K^T) V ("Whisper: Trace One Encoder Tensor into Every
// Decoder Layer", "View 2": one query token, all key tokens, head_dim 64), with
// the SplitKV lazy softmax and its merge ("Caso de estudio: WhisperKit", §3).
//
// A single encoder memory (Whisper-Tiny: 24 rows, Whisper-Base: 48 rows of 1500
// keys) is only ~600-1200 chunks of 64 keys: on 152 SMs a step is then a launch,
// a few copies and a merge, and the persistent kernel's costs -- one copy-issuing
// thread per CTA (bulk copies issued by one thread are processed one after
// another, ~0.23 us each), split rows merged through global partials and an
// arrival counter -- are the step. This kernel is shaped for that regime:
//
//  * Each row gets a cluster of C CTAs; CTA r of the cluster takes keys
//    [r*kl/C, (r+1)*kl/C) of the row. C is the largest size up to 8 for which
//    every row's cluster is resident at once (the occupancy query: clusters are
//    placed inside a GPC, so 3 or 6 CTAs per cluster can leave SMs idle and start
//    a second wave), with 6 warps per CTA when that still allows C = 8, else 4.
//  * Inside a CTA every warp owns its own 2-stage ring of 8 KB stages (16 fp32 /
//    32 bf16 keys of K and V) and issues its own copies, K and V from two lanes
//    (one thread's bulk copies are processed one after another): warp w takes
//    the sub-chunks w, w + W, w + 2W, ... of the CTA's share. Scores: a bf16 key
//    per lane, an fp32 key per lane pair (32 channels each, one shuffle), the
//    16-byte slices read in an order rotated by key so that the warp's reads are
//    conflict-free; P.V with two channels per lane.
//  * Each warp keeps its own online-softmax state (base 2, q pre-scaled by
//    scale * log2 e); the warps' states are merged in shared memory, and the
//    CTAs' states through distributed shared memory into the cluster's rank 0,
//    which writes the row. No global workspace, no atomics, no partials.
//  * Programmatic dependent launch: the rings are filled before the grid
//    dependency wait (the cache and key_len are inputs no decode writes); q is
//    read and out written only after it.
//  * Keys t >= key_len[b] are never copied; a row without keys writes zeros.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>

#include "cxa.h"
#include "internal.h"
#include "chunk_stream.cuh"
#include "cluster.cuh"
#include "ptx.cuh"

namespace cxa {
namespace {

constexpr int kDh = 64;
constexpr int kStages = 2;               // per warp
constexpr int kMaxCluster = 8;           // portable cluster size
constexpr int kStateFloats = 68;         // m, s, 2 pad, acc[64]

struct RowsParams {
  const float* Q;
  const uint8_t* Kc;
  const uint8_t* Vc;
  const int* key_len;
  float* out;
  unsigned int* status;
  int T, LH, LHc, lh0;
  int key_len_add;
  float qscale;
};

template <bool kBF16, int W>
struct RowsTraits {
  static constexpr int kRowBytes = kDh * (kBF16 ? 2 : 4);       // 128 / 256
  static constexpr int kSub = kBF16 ? 32 : 16;                   // keys per sub-chunk
  static constexpr int kHalfBytes = kSub * kRowBytes;            // K (or V) of a sub-chunk: 4 KB
  static constexpr int kStageBytes = 2 * kHalfBytes;             // 8 KB
  static constexpr int kRingBytes = W * kStages * kStageBytes;
  static constexpr int kThreads = W * 32;
};

__device__ __forceinline__ void allow_dependent_launch_rows() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prior_grid_rows() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

template <bool kBF16, int W>
__global__ void __launch_bounds__(W * 32) decode_rows_kernel(const RowsParams p) {
  using R = RowsTraits<kBF16, W>;
  constexpr int G = R::kSub;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                                                       // [W][S][K | V]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + R::kRingBytes);         // [W][S] full barriers
  float* s_q = reinterpret_cast<float*>(bars + W * kStages);                  // [64] scaled query
  float* s_warp = s_q + kDh;                                                  // [W][68] warp states
  float* s_cta = s_warp + W * kStateFloats;                                   // [kMaxCluster][68] (rank 0)
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_cta + kMaxCluster * kStateFloats);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  allow_dependent_launch_rows();

  uint32_t nctarank;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(nctarank));
  const int csize = static_cast<int>(nctarank);
  const int rank = static_cast<int>(cluster_rank());
  const int row = static_cast<int>(blockIdx.x) / csize;                       // (slot, layer-head) row of the call
  const int b = row / p.LH;
  const int lh = row - b * p.LH;
  const long long crow = static_cast<long long>(b) * p.LHc + p.lh0 + lh;     // cache row
  const int kl = min(max(__ldg(p.key_len + b) + p.key_len_add, 0), p.T);      // (its latency overlaps the set-up)

  if (threadIdx.x < W * kStages) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
  if (threadIdx.x == 0) *s_abort = 0;
  if (threadIdx.x < W * kStages) fence_mbar_init();
  __syncthreads();
  // every CTA of the cluster has started before any write to another's shared
  // memory (the matching wait comes just before the state exchange)
  cluster_arrive();

  const int k0 = static_cast<int>(static_cast<long long>(rank) * kl / csize);
  const int k1 = static_cast<int>(static_cast<long long>(rank + 1) * kl / csize);
  const int share = k1 - k0;
  const int nsub = (share + G - 1) / G;                                     // sub-chunks of this CTA
  const int mine = warp < nsub ? (nsub - warp + W - 1) / W : 0;             // sub-chunks of this warp
  const uint8_t* Kbase = p.Kc + (static_cast<size_t>(crow) * p.T + k0) * R::kRowBytes;
  const uint8_t* Vbase = p.Vc + (static_cast<size_t>(crow) * p.T + k0) * R::kRowBytes;
  const uint64_t pol = policy_evict_first();
  uint8_t* my_ring = ring + static_cast<size_t>(warp) * kStages * R::kStageBytes;
  uint64_t* my_bars = bars + warp * kStages;

  // Sub-chunk i of this warp (its i-th) goes to stage i % S: lane `kl_lane` arms the
  // barrier and copies K, lane kl_lane + 1 copies V. Called by the whole warp.
  auto issue = [&](int i, int k_lane) {
    const bool act = lane == k_lane || lane == k_lane + 1;
    const int t0 = (warp + i * W) * G;
    const uint32_t bytes = static_cast<uint32_t>(min(G, share - t0)) * R::kRowBytes;
    const int s = i % kStages;
    const uint32_t full = smem_u32(&my_bars[s]);
    const uint32_t dst = smem_u32(my_ring + s * R::kStageBytes);
    if (lane == k_lane) mbar_arrive_expect_tx(full, 2 * bytes);
    __syncwarp();
    if (act && lane == k_lane) bulk_g2s_hint(dst, Kbase + static_cast<size_t>(t0) * R::kRowBytes, bytes, full, pol);
    if (act && lane == k_lane + 1)
      bulk_g2s_hint(dst + R::kHalfBytes, Vbase + static_cast<size_t>(t0) * R::kRowBytes, bytes, full, pol);
  };
  // the first stages before the grid dependency wait, each from its own lane pair
  const int npre = mine < kStages ? mine : kStages;
  for (int i = 0; i < kStages; ++i)
    if (i < npre) issue(i, 2 * i);
  int issued = npre;

  // q (and out) may belong to the previous grid on the stream
  wait_prior_grid_rows();
  if (threadIdx.x < kDh / 4) {
    // an L2 load: the previous grid may have just written q
    const float4 v = __ldcg(reinterpret_cast<const float4*>(p.Q + static_cast<long long>(row) * kDh) + threadIdx.x);
    reinterpret_cast<float4*>(s_q)[threadIdx.x] =
        make_float4(v.x * p.qscale, v.y * p.qscale, v.z * p.qscale, v.w * p.qscale);
  }
  __syncthreads();

  float m = -INFINITY, ssum = 0.f, a0 = 0.f, a1 = 0.f;   // lane owns channels 2*lane, 2*lane + 1
  bool ok = true;
  for (int i = 0; i < mine; ++i) {
    const int s = i % kStages;
    const uint32_t parity = static_cast<uint32_t>((i / kStages) & 1);
    const bool got = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(&my_bars[s]), parity, s_abort));
    if (ok && !got) {                    // warp-uniform: the whole warp stops here
      ok = false;
      if (lane == 0) {
        *s_abort = 1;
        atomicOr(p.status, 1u);
      }
    }
    const int n = min(G, share - (warp + i * W) * G);
    const uint8_t* sK = my_ring + s * R::kStageBytes;
    const uint8_t* sV = sK + R::kHalfBytes;
    if (ok) {
      float sc = 0.f;
      int key;
      if constexpr (kBF16) {
        // a key per lane, 8 slices of 8 channels
        key = lane;
        const uint8_t* krow = sK + lane * R::kRowBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int ch = (c + lane) & 7;
          const uint4 u = *reinterpret_cast<const uint4*>(krow + ch * 16);
          const float4 qa = reinterpret_cast<const float4*>(s_q)[2 * ch];
          const float4 qb = reinterpret_cast<const float4*>(s_q)[2 * ch + 1];
          sc = fmaf(qa.x, __uint_as_float(u.x << 16), sc);
          sc = fmaf(qa.y, __uint_as_float(u.x & 0xFFFF0000u), sc);
          sc = fmaf(qa.z, __uint_as_float(u.y << 16), sc);
          sc = fmaf(qa.w, __uint_as_float(u.y & 0xFFFF0000u), sc);
          sc = fmaf(qb.x, __uint_as_float(u.z << 16), sc);
          sc = fmaf(qb.y, __uint_as_float(u.z & 0xFFFF0000u), sc);
          sc = fmaf(qb.z, __uint_as_float(u.w << 16), sc);
          sc = fmaf(qb.w, __uint_as_float(u.w & 0xFFFF0000u), sc);
        }
      } else {
        // a key per lane pair, each lane 32 channels (8 slices of 4)
        key = lane >> 1;
        const int half = lane & 1;
        const uint8_t* krow = sK + key * R::kRowBytes + half * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int ch = (c + key) & 7;
          const float4 k4 = *reinterpret_cast<const float4*>(krow + ch * 16);
          const float4 q4 = reinterpret_cast<const float4*>(s_q)[half * 8 + ch];
          sc = fmaf(q4.x, k4.x, sc);
          sc = fmaf(q4.y, k4.y, sc);
          sc = fmaf(q4.z, k4.z, sc);
          sc = fmaf(q4.w, k4.w, sc);
        }
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
      }
      const bool valid = key < n;
      const float sv = valid ? sc : -INFINITY;
      const float mnew = fmaxf(m, warp_max(sv));
      const float corr = rescale(m, mnew);                                   // 0 while the state is empty
      m = mnew;
      const float pw = valid ? exp2f(sv - mnew) : 0.f;
      ssum *= corr;
      a0 *= corr;
      a1 *= corr;
      // ---- P.V over the valid keys: p of key k broadcast from its lane
      for (int k = 0; k < n; ++k) {
        const float pk = __shfl_sync(0xffffffffu, pw, kBF16 ? k : 2 * k);
        float v0, v1;
        if constexpr (kBF16) {
          const uint32_t u = *reinterpret_cast<const uint32_t*>(sV + k * R::kRowBytes + lane * 4);
          v0 = __uint_as_float(u << 16);
          v1 = __uint_as_float(u & 0xFFFF0000u);
        } else {
          const float2 v = *reinterpret_cast<const float2*>(sV + k * R::kRowBytes + lane * 8);
          v0 = v.x;
          v1 = v.y;
        }
        ssum += pk;
        a0 = fmaf(pk, v0, a0);
        a1 = fmaf(pk, v1, a1);
      }
    }
    __syncwarp();                        // every lane is done with the stage before it is refilled
    if (ok && i + kStages < mine) {
      issue(i + kStages, 0);
      ++issued;
    }
  }
  if (!ok && lane == 0) {
    // let this warp's copies in flight land before the CTA can exit: on each stage,
    // wait (bounded) for the last phase issued there
    for (int s = 0; s < kStages; ++s) {
      int on_s = 0;
      for (int i = s; i < issued; i += kStages) ++on_s;
      if (on_s > 0) mbar_wait(smem_u32(&my_bars[s]), static_cast<uint32_t>((on_s - 1) & 1));
    }
  }

  // ---- the warps' states -> one per CTA (warp 0), then the cluster's -> rank 0
  float* ws = s_warp + warp * kStateFloats;
  ws[4 + 2 * lane] = a0;
  ws[4 + 2 * lane + 1] = a1;
  if (lane == 0) {
    ws[0] = ok ? m : -INFINITY;
    ws[1] = ok ? ssum : 0.f;
  }
  __syncthreads();
  float M = -INFINITY, S = 0.f, A0 = 0.f, A1 = 0.f;
  if (warp == 0) {
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, s_warp[w * kStateFloats]);
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float f = rescale(s_warp[w * kStateFloats], M);
      S = fmaf(s_warp[w * kStateFloats + 1], f, S);
      A0 = fmaf(s_warp[w * kStateFloats + 4 + 2 * lane], f, A0);
      A1 = fmaf(s_warp[w * kStateFloats + 4 + 2 * lane + 1], f, A1);
    }
  }
  cluster_wait();                        // (pairs with the arrive after the set-up)
  if (warp == 0) {
    // this CTA's state into slot `rank` of the cluster's rank-0 CTA
    float* slot = s_cta + rank * kStateFloats;
    st_dsmem(slot + 4 + 2 * lane, 0, A0);
    st_dsmem(slot + 4 + 2 * lane + 1, 0, A1);
    if (lane == 0) {
      st_dsmem(slot, 0, M);
      st_dsmem(slot + 1, 0, S);
    }
  }
  cluster_sync();                        // every CTA's state has landed in rank 0
  if (rank == 0 && warp == 0) {
    M = -INFINITY;
    for (int r = 0; r < csize; ++r) M = fmaxf(M, s_cta[r * kStateFloats]);
    S = A0 = A1 = 0.f;
    for (int r = 0; r < csize; ++r) {
      const float f = rescale(s_cta[r * kStateFloats], M);
      S = fmaf(s_cta[r * kStateFloats + 1], f, S);
      A0 = fmaf(s_cta[r * kStateFloats + 4 + 2 * lane], f, A0);
      A1 = fmaf(s_cta[r * kStateFloats + 4 + 2 * lane + 1], f, A1);
    }
    const float inv = S > 0.f ? 1.f / S : 0.f;
    reinterpret_cast<float2*>(p.out + static_cast<long long>(row) * kDh)[lane] = make_float2(A0 * inv, A1 * inv);
  }
}

template <bool kBF16, int W>
size_t rows_smem_bytes() {
  using R = RowsTraits<kBF16, W>;
  return static_cast<size_t>(R::kRingBytes) + W * kStages * sizeof(uint64_t) +
         (kDh + W * kStateFloats + kMaxCluster * kStateFloats) * sizeof(float) + 16;
}

template <bool kBF16, int W>
cudaLaunchConfig_t rows_config(int rows, int csize, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(rows * csize));
  cfg.blockDim = dim3(RowsTraits<kBF16, W>::kThreads);
  cfg.dynamicSmemBytes = rows_smem_bytes<kBF16, W>();
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned int>(csize);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// Per device and instance: the shared-memory attribute, and how many clusters of
// each size 1..8 can be resident at once (cudaOccupancyMaxActiveClusters).
struct RowsOccupancy {
  bool ready = false;
  int max_clusters[kMaxCluster + 1] = {};
};

template <bool kBF16, int W>
cudaError_t rows_occupancy(int device, const RowsOccupancy** out) {
  static std::mutex mu;
  static RowsOccupancy table[128];
  if (device < 0 || device >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  RowsOccupancy& o = table[device];
  if (!o.ready) {
    cudaError_t e = cudaFuncSetAttribute(decode_rows_kernel<kBF16, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(rows_smem_bytes<kBF16, W>()));
    if (e != cudaSuccess) return e;
    for (int c = 1; c <= kMaxCluster; ++c) {
      cudaLaunchAttribute attr[2];
      cudaLaunchConfig_t cfg = rows_config<kBF16, W>(c, c, nullptr, attr);
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, decode_rows_kernel<kBF16, W>, &cfg);
      if (e != cudaSuccess) return e;
      o.max_clusters[c] = n;
    }
    o.ready = true;
  }
  *out = &o;
  return cudaSuccess;
}

// The largest cluster size whose `rows` clusters are all resident at once (0: none).
int largest_resident_cluster(const RowsOccupancy& o, int rows) {
  for (int c = kMaxCluster; c >= 1; --c)
    if (o.max_clusters[c] >= rows) return c;
  return 0;
}

template <bool kBF16>
cudaError_t launch_rows(const RowsParams& prm, int rows, const DeviceInfo& dev, cudaStream_t stream, bool* done) {
  *done = false;
  const RowsOccupancy* o6 = nullptr;
  const RowsOccupancy* o4 = nullptr;
  cudaError_t e = rows_occupancy<kBF16, 6>(dev.device, &o6);
  if (e != cudaSuccess) return e;
  e = rows_occupancy<kBF16, 4>(dev.device, &o4);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  // six warps per CTA when clusters of 8 still fit, else four warps and the largest
  // cluster that fits
  if (largest_resident_cluster(*o6, rows) == kMaxCluster) {
    cudaLaunchConfig_t cfg = rows_config<kBF16, 6>(rows, kMaxCluster, stream, attr);
    *done = true;
    return cudaLaunchKernelEx(&cfg, decode_rows_kernel<kBF16, 6>, prm);
  }
  const int c = largest_resident_cluster(*o4, rows);
  if (c == 0) return cudaSuccess;                                   // does not fit: the caller streams
  cudaLaunchConfig_t cfg = rows_config<kBF16, 4>(rows, c, stream, attr);
  *done = true;
  return cudaLaunchKernelEx(&cfg, decode_rows_kernel<kBF16, 4>, prm);
}

}  // namespace

bool decode_rows_eligible(int rows, int T, int num_sms, int policy) {
  if (policy == CXA_DECODE_STREAM || rows < 1) return false;
  if (policy == CXA_DECODE_ROWS) return true;
  // automatic choice: short streams only, a few 64-key chunks per SM in all
  const long long chunks = static_cast<long long>(rows) * ((T + 63) / 64);
  return rows <= 2 * num_sms && chunks <= 8LL * num_sms;
}

cudaError_t launch_decode_rows(const DecodeLaunch& a, const DeviceInfo& dev, cudaStream_t stream, bool* done) {
  RowsParams prm;
  prm.Q = a.Q;
  prm.Kc = static_cast<const uint8_t*>(a.Kc);
  prm.Vc = static_cast<const uint8_t*>(a.Vc);
  prm.key_len = a.key_len;
  prm.out = a.out;
  prm.status = dev.status_word;
  prm.T = a.T;
  prm.LH = a.nl * a.H;
  prm.LHc = a.L * a.H;
  prm.lh0 = a.l0 * a.H;
  prm.key_len_add = a.key_len_add;
  prm.qscale = a.scale * 1.4426950408889634f;   // scale * log2(e)
  const int rows = a.B * a.nl * a.H;
  const cudaError_t e = a.cache_bf16 ? launch_rows<true>(prm, rows, dev, stream, done)
                                     : launch_rows<false>(prm, rows, dev, stream, done);
  if (e == cudaSuccess && *done) count_launches(1);
  return e;
}

}  // namespace cxa
