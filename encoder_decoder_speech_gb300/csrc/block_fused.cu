// One decoder layer's cross-attention block for one decode step as ONE kernel
// ("Whisper: Trace One Encoder Tensor into Every Decoder Layer", "The concept":
// Q_l = decoder_hidden_l x WQ_l against the cached K_l/V_l; the decoder body's
// cross_attn_norm -> cross_q_proj -> cross_attn -> cross_out_proj):
//
//   h = LayerNorm(x_b);  q_bh = h x WQ[:, head h] + bQ
//   o_bh = softmax(scale q_bh . K_bh^T) V_bh over the slot's valid keys
//   x_b += concat_h(o_bh) x WO + bO
//
// A thread-block cluster of H CTAs per slot b, CTA h of the cluster owning head h
// (H <= 8: a portable cluster). Each CTA
//   * streams its (b, layer, h) K/V row through a 16-stage bulk-copy ring (24 fp32 /
//     32 bf16 keys of K and V per stage) from its first instruction (no earlier
//     kernel writes the cache); chunk i belongs to warp i % 8 alone, which waits
//     for it, runs it through its lane groups' softmax states and refills the
//     stage with chunk i + 16, so no warp waits for another within the loop;
//   * loads its 64-column slice of WQ into registers before waiting on the
//     previous grid (programmatic dependent launch), then normalises x_b and
//     projects its head's query;
//   * runs the online softmax over the ring (8 warps, a 16-byte slice of a key row
//     per lane; each lane group takes its keys of a chunk together: scores, one
//     rescale of its running max / sum / accumulator, then the V rows; the groups
//     merge once at the end), loading its WO slice into registers meanwhile;
//   * publishes o_bh in shared memory, gathers the slot's whole attention row
//     from its cluster peers (distributed shared memory), and writes columns
//     [64h, 64h + 64) of x_b = x_b + a x WO + bO.
// Nothing goes through global memory between the four steps, and one launch
// replaces three.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>

#include "chunk_stream.cuh"
#include "cluster.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace cxa {
namespace {

constexpr int kDh = 64;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers;
// Ring shape (compile-time; the defaults were chosen by timing on GB300).
#ifndef CXA_BLOCK_STAGES
#define CXA_BLOCK_STAGES 16
#endif
#ifndef CXA_BLOCK_CHUNK_F32
#define CXA_BLOCK_CHUNK_F32 24
#endif
#ifndef CXA_BLOCK_CHUNK_BF16
#define CXA_BLOCK_CHUNK_BF16 32
#endif
constexpr int kStages = CXA_BLOCK_STAGES;
static_assert(kStages % kConsumerWarps == 0, "each warp owns kStages / 8 stages");
constexpr int kMaxHeads = 8;                       // portable cluster size
constexpr int kMaxD = kMaxHeads * kDh;
constexpr int kRowGroups = 16;                     // projection: 16 groups of d/16 input rows
constexpr int kMaxRowsPerGroup = kMaxD / kRowGroups;   // 32

template <bool kBF16>
struct FusedTraits {
  static constexpr int kElem = kBF16 ? 2 : 4;
  static constexpr int kRowBytes = kDh * kElem;              // 256 / 128
  static constexpr int kChunkKeys = kBF16 ? CXA_BLOCK_CHUNK_BF16 : CXA_BLOCK_CHUNK_F32;   // keys per stage
  static constexpr int kTileBytes = kChunkKeys * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;         // K then V
  static constexpr int kLanesPerKey = kBF16 ? 8 : 16;        // one 16-byte slice of a row per lane
  static constexpr int kKeysPerPass = 32 / kLanesPerKey;     // keys per warp per pass
  static constexpr int kChanPerLane = 16 / kElem;            // 4 / 8 channels
  static constexpr int kGroups = kConsumerWarps * kKeysPerPass;   // softmax states per CTA
  static constexpr int kPasses = kChunkKeys / kKeysPerPass;  // passes of one warp over a chunk
  static_assert(kPasses * kKeysPerPass == kChunkKeys, "chunk = whole passes");
};

struct FusedParams {
  const uint8_t* Kc;
  const uint8_t* Vc;
  float* x;
  const float* gamma;
  const float* beta;
  const float* WQ;
  const float* bQ;
  const float* WO;
  const float* bO;
  const int* key_len;
  float* att;          // [B][d] attention rows (kGather == false)
  unsigned int* status;
  int T, L, H, layer, d;
  float eps, qscale;   // qscale = scale * log2(e)
};

__device__ __forceinline__ void consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// The 16-byte slice of a cached row at byte offset off, as kChanPerLane floats.
template <bool kBF16>
__device__ __forceinline__ void load_slice(const uint8_t* p, float (&v)[FusedTraits<kBF16>::kChanPerLane]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  if constexpr (kBF16) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  } else {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
  }
}

// (n, mean, M2) <- the moments of the union of two disjoint sets of values, M2 being
// the sum of squared deviations from the mean (Chan, Golub and LeVeque's pairwise update).
__device__ __forceinline__ void merge_moments(float& n, float& mean, float& m2, float nb, float mb, float m2b) {
  if (nb == 0.f) return;
  if (n == 0.f) {
    n = nb;
    mean = mb;
    m2 = m2b;
    return;
  }
  const float nn = n + nb;
  const float dl = mb - mean;
  const float f = nb / nn;
  mean = fmaf(dl, f, mean);
  m2 = m2 + m2b + dl * dl * n * f;
  n = nn;
}

// y[c] = sum_i in[i] W[i][col0 + c] for c < 64, by the 256 consumer threads: thread
// (row group rg = t / 16, column quad cq = t % 16) owns rows [rg R, rg R + R) of the
// slice, held in w (R = d / 16 rows); the 16 partial quads meet in red[16][64].
__device__ __forceinline__ void project_partial(const float4 (&w)[kMaxRowsPerGroup], const float* in, int R, int rg,
                                                int cq, float* red) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kMaxRowsPerGroup; ++j) {
    if (j < R) {
      const float h = in[rg * R + j];
      acc.x = fmaf(h, w[j].x, acc.x);
      acc.y = fmaf(h, w[j].y, acc.y);
      acc.z = fmaf(h, w[j].z, acc.z);
      acc.w = fmaf(h, w[j].w, acc.w);
    }
  }
  *reinterpret_cast<float4*>(red + rg * kDh + 4 * cq) = acc;
}
__device__ __forceinline__ void load_weights(float4 (&w)[kMaxRowsPerGroup], const float* W, int d, int col0, int R,
                                             int rg, int cq) {
#pragma unroll
  for (int j = 0; j < kMaxRowsPerGroup; ++j)
    w[j] = j < R ? __ldg(reinterpret_cast<const float4*>(W + static_cast<size_t>(rg * R + j) * d + col0) + cq)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
}

// kGather: the whole block in one launch (a cluster of H CTAs per slot gathers the
// attention row and applies WO). Otherwise each CTA stops at its attention output,
// written to att[b][64h + c], and the out projection is a separate GEMV launch:
// that form needs no cluster, so all B*H CTAs are resident at once even when B
// clusters of H would not be.
template <bool kBF16, bool kGather>
__global__ void __maxnreg__(224) fused_block_kernel(const FusedParams p) {
  using R_ = FusedTraits<kBF16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  float* s_x = reinterpret_cast<float*>(ring + kStages * R_::kStageBytes);   // [d] x_b as read
  float* s_h = s_x + kMaxD;                               // [d] LayerNorm(x_b), later the gathered attention row
  float* s_red = s_h + kMaxD;                             // [16][64] projection partials
  float* s_q = s_red + kRowGroups * kDh;                  // [64] scaled query
  float* s_o = s_q + kDh;                                 // [64] this head's attention output (read by peers)
  float* s_st = s_o + kDh;                                // [kGroups][66] softmax states
  float* s_stat = s_st + R_::kGroups * (kDh + 2);         // [8][3] LayerNorm moments per warp
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_stat + 32);   // full[kStages]
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + kStages);
  int* s_last = const_cast<int*>(s_abort) + 1;             // [kStages] last chunk issued into stage s

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int h = blockIdx.x;                               // head = column block = cluster rank
  const int b = blockIdx.y;
  const int d = p.d;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      s_last[s] = -1;
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int kl = min(max(__ldg(p.key_len + b), 0), p.T);
  const int nch = (kl + R_::kChunkKeys - 1) / R_::kChunkKeys;
  const size_t row_off = (static_cast<size_t>(b) * p.L * p.H + static_cast<size_t>(p.layer) * p.H + h) *
                         static_cast<size_t>(p.T) * R_::kRowBytes;
  const int R = d / kRowGroups;                           // projection: input rows per row group
  const int rg = tid >> 4, cq = tid & 15;
  float4 w[kMaxRowsPerGroup];                             // WQ slice, then the WO slice

  // chunk i of the row into stage i % kStages; the K/V rows are read once per step,
  // so they go in L2 as evict-first and the layer's weights stay resident
  const uint64_t pol = policy_evict_first();
  auto issue = [&](int i) {
    const int s = i % kStages;
    const int n = min(R_::kChunkKeys, kl - i * R_::kChunkKeys);
    const uint32_t bytes = static_cast<uint32_t>(n) * R_::kRowBytes;
    const size_t off = row_off + static_cast<size_t>(i) * R_::kTileBytes;
    const uint32_t full = smem_u32(&bars[s]);
    const uint32_t dst = smem_u32(ring + s * R_::kStageBytes);
    s_last[s] = i;
    mbar_arrive_expect_tx(full, 2 * bytes);
    bulk_g2s_hint(dst, p.Kc + off, bytes, full, pol);
    bulk_g2s_hint(dst + R_::kTileBytes, p.Vc + off, bytes, full, pol);
  };
  // chunk i belongs to warp i % 8 alone: that warp waits for it, computes it and
  // refills its stage with chunk i + kStages (kStages is a multiple of 8)
  if (lane == 0)
    for (int i = warp; i < min(nch, kStages); i += kConsumerWarps) issue(i);
  {
    // ------------------------------------------------------------ consumers
    load_weights(w, p.WQ, d, h * kDh, R, rg, cq);          // no earlier kernel writes the weights
    float gv[kMaxD / kConsumers], bv[kMaxD / kConsumers];   // this thread's LayerNorm gain and bias
#pragma unroll
    for (int e = 0; e < kMaxD / kConsumers; ++e) {
      const int i = tid + e * kConsumers;
      gv[e] = p.gamma && i < d ? __ldg(p.gamma + i) : 1.f;
      bv[e] = p.beta && i < d ? __ldg(p.beta + i) : 0.f;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");     // x may come from the previous grid

    // ---- h = LayerNorm(x_b), biased variance. One pass: each thread's elements
    //      i = tid, tid + 256 give a (count, mean, squared deviations) triple; the
    //      triples merge pairwise (Chan, Golub and LeVeque's update) across the warp
    //      by shuffles, then across the eight warps through shared memory.
    const float* xb = p.x + static_cast<size_t>(b) * d;
    float xv[kMaxD / kConsumers];
    float cn = 0.f, cm = 0.f, c2 = 0.f;
#pragma unroll
    for (int e = 0; e < kMaxD / kConsumers; ++e) {
      const int i = tid + e * kConsumers;
      xv[e] = i < d ? xb[i] : 0.f;
      if (i < d) {
        s_x[i] = xv[e];
        cn += 1.f;
        const float dl = xv[e] - cm;
        cm += dl / cn;
        c2 = fmaf(dl, xv[e] - cm, c2);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float on = __shfl_xor_sync(0xffffffffu, cn, off);
      const float om = __shfl_xor_sync(0xffffffffu, cm, off);
      const float o2 = __shfl_xor_sync(0xffffffffu, c2, off);
      merge_moments(cn, cm, c2, on, om, o2);
    }
    if (lane == 0) {
      s_stat[3 * warp] = cn;
      s_stat[3 * warp + 1] = cm;
      s_stat[3 * warp + 2] = c2;
    }
    consumer_barrier();
    float n_all = s_stat[0], mean = s_stat[1], m2 = s_stat[2];
#pragma unroll
    for (int k = 1; k < kConsumerWarps; ++k) merge_moments(n_all, mean, m2, s_stat[3 * k], s_stat[3 * k + 1], s_stat[3 * k + 2]);
    const float rstd = rsqrtf(m2 / static_cast<float>(d) + p.eps);
#pragma unroll
    for (int e = 0; e < kMaxD / kConsumers; ++e) {
      const int i = tid + e * kConsumers;
      if (i < d) s_h[i] = fmaf((xv[e] - mean) * rstd, gv[e], bv[e]);
    }
    consumer_barrier();

    // ---- q_bh = h x WQ[:, head] + bQ, pre-scaled by scale * log2(e)
    project_partial(w, s_h, R, rg, cq, s_red);
    consumer_barrier();
    if (tid < kDh) {
      float q = p.bQ ? __ldg(p.bQ + h * kDh + tid) : 0.f;
#pragma unroll
      for (int k = 0; k < kRowGroups; ++k) q += s_red[k * kDh + tid];
      s_q[tid] = q * p.qscale;
    }
    consumer_barrier();
    // the out-projection slice: its loads run under the attention loop
    if constexpr (kGather) load_weights(w, p.WO, d, h * kDh, R, rg, cq);

    // ---- attention over the ring: warp wp takes chunks wp, wp + 8, ...; within a
    //      chunk its lane group u takes keys u, u + KPP, ... (one softmax state each)
    constexpr int LPK = R_::kLanesPerKey, CPL = R_::kChanPerLane, KPP = R_::kKeysPerPass;
    const int u = lane / LPK, sl = lane % LPK;             // key within the pass, 16-byte slice
    float qv[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) qv[c] = s_q[sl * CPL + c];
    float m = -INFINITY, l = 0.f, acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
    bool ok = true;
    for (int i = warp; i < nch; i += kConsumerWarps) {
      const int s = i % kStages;
      if (ok && !mbar_wait(smem_u32(&bars[s]), static_cast<uint32_t>((i / kStages) & 1), s_abort)) {
        ok = false;
        *s_abort = 1;
        atomicOr(p.status, 1u);
      }
      const int n = min(R_::kChunkKeys, kl - i * R_::kChunkKeys);
      const uint8_t* kt = ring + s * R_::kStageBytes;
      const uint8_t* vt = kt + R_::kTileBytes;
      // the chunk's scores for this lane group first (independent shuffle chains),
      // then one rescale of the running state per chunk, then the weighted V rows
      float sc[R_::kPasses];
#pragma unroll
      for (int ps = 0; ps < R_::kPasses; ++ps) {
        const int k = ps * KPP + u;
        const bool valid = k < n && ok;
        float kv[CPL];
        load_slice<kBF16>(kt + (valid ? k : 0) * R_::kRowBytes + sl * 16, kv);
        float v = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) v = fmaf(qv[c], kv[c], v);
        sc[ps] = v;
      }
#pragma unroll
      for (int off = LPK / 2; off >= 1; off >>= 1)
#pragma unroll
        for (int ps = 0; ps < R_::kPasses; ++ps) sc[ps] += __shfl_xor_sync(0xffffffffu, sc[ps], off);
      float cm = -INFINITY;
#pragma unroll
      for (int ps = 0; ps < R_::kPasses; ++ps) {
        const int k = ps * KPP + u;
        if (k >= n || !ok) sc[ps] = -INFINITY;
        cm = fmaxf(cm, sc[ps]);
      }
      if (cm != -INFINITY) {
        const float mn = fmaxf(m, cm);
        const float corr = rescale(m, mn);
        l *= corr;
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] *= corr;
        m = mn;
#pragma unroll
        for (int ps = 0; ps < R_::kPasses; ++ps) {
          const int k = ps * KPP + u;
          if (sc[ps] != -INFINITY) {
            float vv[CPL];
            load_slice<kBF16>(vt + k * R_::kRowBytes + sl * 16, vv);
            const float pr = exp2f(sc[ps] - mn);
            l += pr;
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = fmaf(pr, vv[c], acc[c]);
          }
        }
      }
      __syncwarp();                                        // every lane is done with the stage
      if (lane == 0 && i + kStages < nch && *s_abort == 0) issue(i + kStages);
    }
    // ---- merge the kGroups states: o = sum_g acc_g 2^(m_g - M) / sum_g l_g 2^(m_g - M)
    const int gidx = warp * KPP + u;
    float* st = s_st + gidx * (kDh + 2);
    if (sl == 0) {
      st[0] = m;
      st[1] = l;
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) st[2 + sl * CPL + c] = acc[c];
    consumer_barrier();
    // every warp has left the loop: after a timeout, let the copies still in flight land
    if (*s_abort != 0 && tid == 0)
      for (int s = 0; s < kStages; ++s)
        if (s_last[s] >= 0) mbar_wait(smem_u32(&bars[s]), static_cast<uint32_t>((s_last[s] / kStages) & 1));
    if (tid < kDh) {
      float M = -INFINITY;
      for (int g = 0; g < R_::kGroups; ++g) M = fmaxf(M, s_st[g * (kDh + 2)]);
      float L = 0.f, A = 0.f;
      for (int g = 0; g < R_::kGroups; ++g) {
        const float f = rescale(s_st[g * (kDh + 2)], M);
        L = fmaf(s_st[g * (kDh + 2) + 1], f, L);
        A = fmaf(s_st[g * (kDh + 2) + 2 + tid], f, A);
      }
      const float o = (L > 0.f && ok) ? A / L : 0.f;
      if constexpr (kGather)
        s_o[tid] = o;
      else
        p.att[static_cast<size_t>(b) * d + h * kDh + tid] = o;
    }
  }
  if constexpr (!kGather) return;
  // ---- every head's output of this slot: from the cluster peers' shared memory
  cluster_sync();
  for (int i = tid; i < p.H * kDh; i += kConsumers)
    s_h[i] = ld_dsmem(s_o + (i % kDh), static_cast<uint32_t>(i / kDh));
  cluster_sync();                                          // peers may leave once everyone has gathered
  {
    // ---- x_b[64h + c] += a x WO[:, 64h + c] + bO (w holds the WO slice)
    project_partial(w, s_h, R, rg, cq, s_red);
    consumer_barrier();
    if (tid < kDh) {
      const int j = h * kDh + tid;
      float y = s_x[j] + (p.bO ? __ldg(p.bO + j) : 0.f);
#pragma unroll
      for (int k = 0; k < kRowGroups; ++k) y += s_red[k * kDh + tid];
      if (*s_abort == 0) p.x[static_cast<size_t>(b) * d + j] = y;
    }
  }
}

template <bool kBF16>
size_t fused_smem_bytes() {
  using R_ = FusedTraits<kBF16>;
  return 128 + static_cast<size_t>(kStages) * R_::kStageBytes +
         (2 * kMaxD + kRowGroups * kDh + 2 * kDh + R_::kGroups * (kDh + 2) + 32) * sizeof(float) +
         kStages * (sizeof(uint64_t) + sizeof(int)) + 16;
}

template <bool kBF16, bool kGather>
cudaError_t launch_fused(const FusedParams& prm, int B, const DeviceInfo& dev, cudaStream_t stream) {
  static std::mutex mu;
  static bool attr_set[128] = {};
  const size_t smem = fused_smem_bytes<kBF16>();
  {
    std::lock_guard<std::mutex> lock(mu);
    const int dv = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
    if (!attr_set[dv]) {
      cudaError_t e = cudaFuncSetAttribute(fused_block_kernel<kBF16, kGather>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_set[dv] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.H, B, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = prm.H;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kGather ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fused_block_kernel<kBF16, kGather>, prm);
}

// Clusters of H CTAs of the one-launch block that fit on the device at once
// (queried once per device, dtype and H).
template <bool kBF16>
int resident_clusters(int H, const DeviceInfo& dev) {
  static std::mutex mu;
  static int cache[128][kMaxHeads + 1] = {};
  const int dv = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dv][H] == 0) {
    const size_t smem = fused_smem_bytes<kBF16>();
    int n = 0;
    if (cudaFuncSetAttribute(fused_block_kernel<kBF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(H, 1, 1);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = H;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, fused_block_kernel<kBF16, true>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cache[dv][H] = n > 0 ? n : -1;
  }
  return cache[dv][H];
}

}  // namespace

bool fused_block_supported(int H, int dh) { return dh == kDh && H >= 1 && H <= kMaxHeads; }

cudaError_t launch_block_fused(const BlockLaunch& a, float* att, bool* gathered, const DeviceInfo& dev,
                               cudaStream_t stream) {
  FusedParams prm;
  prm.Kc = static_cast<const uint8_t*>(a.Kc);
  prm.Vc = static_cast<const uint8_t*>(a.Vc);
  prm.x = a.x;
  prm.gamma = a.gamma;
  prm.beta = a.beta;
  prm.WQ = a.WQ;
  prm.bQ = a.bQ;
  prm.WO = a.WO;
  prm.bO = a.bO;
  prm.key_len = a.key_len;
  prm.att = att;
  prm.status = dev.status_word;
  prm.T = a.T;
  prm.L = a.L;
  prm.H = a.H;
  prm.layer = a.layer;
  prm.d = a.H * kDh;
  prm.eps = a.eps;
  prm.qscale = a.scale * 1.4426950408889634f;
  const int fit = a.cache_bf16 ? resident_clusters<true>(a.H, dev) : resident_clusters<false>(a.H, dev);
  *gathered = fit >= a.B;
  cudaError_t e;
  if (*gathered)
    e = a.cache_bf16 ? launch_fused<true, true>(prm, a.B, dev, stream) : launch_fused<false, true>(prm, a.B, dev, stream);
  else
    e = a.cache_bf16 ? launch_fused<true, false>(prm, a.B, dev, stream)
                     : launch_fused<false, false>(prm, a.B, dev, stream);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace cxa
