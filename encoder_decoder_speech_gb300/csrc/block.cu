// The cross-attention block of one decoder layer for one decode step, around
// the cached-K/V attention ("Whisper: Trace One Encoder Tensor into Every
// Decoder Layer", "The concept": Q_l = decoder_hidden_l x WQ_l, and the decoder
// body's cross_attn_norm -> cross_q_proj -> cross_attn -> cross_out_proj):
//
//   h = LayerNorm(x)                 (per slot, over d; gamma, beta, eps)
//   q = h x WQ + bQ                  [B][d] = [B][H][64]
//   a = attention of q over layer l's cached K/V      (decode_stream_kernel)
//   x = x + a x WO + bO              (residual add, in place)
//
// Both projections are one kernel: out[b][j] = sum_i norm(in)[b][i] W[i][j]
// (+ bias, + residual), over a grid of (32-column tile, 1/8 of d_in, 16-slot
// block) CTAs. The 8 CTAs that share a column tile form a thread-block cluster:
// each multiplies its d_in slice, and cluster rank 0 adds the 8 partial tiles
// straight out of its peers' shared memory (distributed shared memory) and
// writes the result: a deterministic split-K with one weight read. Every CTA
// loads its weight tile into registers before waiting on the previous grid
// (programmatic dependent launch), so weight traffic overlaps the previous
// kernel's tail; and every CTA lets the next grid launch early, so the decode
// that follows starts streaming its K/V while the projection finishes.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "cluster.cuh"
#include "internal.h"

namespace cxa {
namespace {

constexpr int kRowsPerCta = 16;                 // slots per CTA (grid z covers B)
constexpr int kColsPerCta = 32;                 // output columns per CTA
constexpr int kCluster = 8;                     // CTAs along d_in = cluster size
constexpr int kGemvThreads = 256;
constexpr int kColQuads = kColsPerCta / 4;      // 8 threads cover a 32-column row (float4 each)
constexpr int kRowGroups = kGemvThreads / kColQuads;   // 32 row groups
constexpr int kMaxSlice = 160;                  // d_in rows per CTA (d <= 1280)

// out[b][j] = (residual ? residual[b][j] : 0) + (bias ? bias[j] : 0)
//             + sum_i norm(in)[b][i] * W[i][j]
// norm = LayerNorm(gamma, beta, eps) when kLayerNorm, identity otherwise.
// out may alias residual (each output element reads only its own residual).
template <bool kLayerNorm>
__global__ void __launch_bounds__(kGemvThreads)
    cluster_gemv_kernel(const float* in, const float* __restrict__ gamma, const float* __restrict__ beta,
                        float eps, const float* __restrict__ W, const float* __restrict__ bias,
                        const float* residual, float* out, int B, int d) {
  // dynamic: the staged input rows, [kRowsPerCta][d] (LayerNorm needs whole rows)
  // or [kRowsPerCta][d / kCluster] (this CTA's d_in slice only)
  extern __shared__ float4 s_dyn[];
  float* s_rows = reinterpret_cast<float*>(s_dyn);
  __shared__ float s_in[kRowsPerCta][kMaxSlice];              // this CTA's d_in slice of the (normalised) rows
  __shared__ float s_mean[kRowsPerCta], s_rstd[kRowsPerCta];
  __shared__ float s_part[kGemvThreads / 32][kRowsPerCta][kColsPerCta];   // per-warp partials
  __shared__ float s_tile[kRowsPerCta][kColsPerCta];          // this CTA's partial tile (read by rank 0)

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = blockIdx.x * kColsPerCta;
  const uint32_t rank = cluster_rank();                       // == blockIdx.y: the d_in slice
  const int slice = d / kCluster;
  const int i0 = static_cast<int>(rank) * slice;
  const int r0 = blockIdx.z * kRowsPerCta;
  const int nr = min(kRowsPerCta, B - r0);
  const int cq = tid % kColQuads, rg = tid / kColQuads;

  // weights first: nothing earlier in the stream writes them
  constexpr int kMaxPer = kMaxSlice / kRowGroups;             // 5 rows per thread at d = 1280
  float4 w[kMaxPer];
#pragma unroll
  for (int m = 0; m < kMaxPer; ++m) {
    const int i = rg + m * kRowGroups;
    w[m] = i < slice ? __ldg(reinterpret_cast<const float4*>(W + static_cast<size_t>(i0 + i) * d + j0) + cq)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");          // the rows may come from the previous grid

  // stage the input rows with every thread's 16-byte loads in flight at once
  const int width = kLayerNorm ? d : slice;                   // floats per staged row
  const int first = kLayerNorm ? 0 : i0;
  const int v4 = width / 4;
  const float4* in4 = reinterpret_cast<const float4*>(in);
#pragma unroll 4
  for (int idx = tid; idx < nr * v4; idx += kGemvThreads) {
    const int r = idx / v4, c = idx - r * v4;
    s_dyn[idx] = in4[(static_cast<size_t>(r0 + r) * d + first) / 4 + c];
  }
  __syncthreads();
  if constexpr (kLayerNorm) {
    for (int r = warp; r < nr; r += kGemvThreads / 32) {      // whole-row statistics from shared memory
      const float* row = s_rows + r * d;
      float sum = 0.f;
      for (int i = lane; i < d; i += 32) sum += row[i];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      const float mean = sum / static_cast<float>(d);
      float v = 0.f;
      for (int i = lane; i < d; i += 32) {
        const float c = row[i] - mean;
        v = fmaf(c, c, v);
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) {
        s_mean[r] = mean;
        s_rstd[r] = rsqrtf(v / static_cast<float>(d) + eps);
      }
    }
    __syncthreads();
  }
  for (int idx = tid; idx < kRowsPerCta * slice; idx += kGemvThreads) {
    const int r = idx / slice, i = idx - r * slice;
    float v = 0.f;
    if (r < nr) {
      if constexpr (kLayerNorm) {
        const float g = gamma ? __ldg(gamma + i0 + i) : 1.f;
        const float bb = beta ? __ldg(beta + i0 + i) : 0.f;
        v = fmaf((s_rows[r * d + i0 + i] - s_mean[r]) * s_rstd[r], g, bb);
      } else {
        v = s_rows[r * slice + i];
      }
    }
    s_in[r][i] = v;
  }
  __syncthreads();

  float acc[kRowsPerCta][4];
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
#pragma unroll
  for (int m = 0; m < kMaxPer; ++m) {
    const int i = rg + m * kRowGroups;
    if (i < slice) {
#pragma unroll
      for (int r = 0; r < kRowsPerCta; ++r) {
        const float h = s_in[r][i];
        acc[r][0] = fmaf(h, w[m].x, acc[r][0]);
        acc[r][1] = fmaf(h, w[m].y, acc[r][1]);
        acc[r][2] = fmaf(h, w[m].z, acc[r][2]);
        acc[r][3] = fmaf(h, w[m].w, acc[r][3]);
      }
    }
  }
  // the 4 row groups of a warp share its column quads: lanes l, l^8, l^16, l^24
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v = acc[r][c];
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      acc[r][c] = v;
    }
  if (lane < kColQuads) {
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) s_part[warp][r][4 * cq + c] = acc[r][c];
  }
  __syncthreads();
  for (int idx = tid; idx < kRowsPerCta * kColsPerCta; idx += kGemvThreads) {
    const int r = idx / kColsPerCta, c = idx - r * kColsPerCta;
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < kGemvThreads / 32; ++k) v += s_part[k][r][c];
    s_tile[r][c] = v;
  }
  cluster_sync();                                             // every CTA's tile is complete
  if (rank == 0) {
    for (int idx = tid; idx < nr * kColsPerCta; idx += kGemvThreads) {
      const int r = idx / kColsPerCta, c = idx - r * kColsPerCta;
      float v = 0.f;
#pragma unroll
      for (int k = 0; k < kCluster; ++k) v += ld_dsmem(&s_tile[r][c], static_cast<uint32_t>(k));
      const size_t o = static_cast<size_t>(r0 + r) * d + j0 + c;
      if (bias) v += __ldg(bias + j0 + c);
      if (residual) v += residual[o];
      out[o] = v;
    }
  }
  cluster_sync();                                             // peers keep their tiles until rank 0 is done
}

template <bool kLayerNorm>
cudaError_t launch_gemv(const float* in, const float* gamma, const float* beta, float eps, const float* W,
                        const float* bias, const float* residual, float* out, int B, int d, int device,
                        cudaStream_t stream) {
  static std::mutex mu;
  static size_t attr_bytes[128] = {};
  const size_t smem = static_cast<size_t>(kRowsPerCta) * (kLayerNorm ? d : d / kCluster) * sizeof(float);
  {
    std::lock_guard<std::mutex> lock(mu);
    const int dv = device >= 0 && device < 128 ? device : 0;
    if (attr_bytes[dv] < smem) {
      cudaError_t e = cudaFuncSetAttribute(cluster_gemv_kernel<kLayerNorm>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_bytes[dv] = smem;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d / kColsPerCta, kCluster, (B + kRowsPerCta - 1) / kRowsPerCta);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = kCluster;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, cluster_gemv_kernel<kLayerNorm>, in, gamma, beta, eps, W, bias, residual,
                                     out, B, d);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t block_workspace_bytes(int B, int T, int H) {
  const size_t rows = align256(static_cast<size_t>(B) * H * 64 * sizeof(float));
  return decode_workspace_bytes(B, T, 1, H, 1) + 2 * rows;
}

cudaError_t launch_block(const BlockLaunch& a, const DeviceInfo& dev, cudaStream_t stream, std::string* msg) {
  const int d = a.H * 64;
  if (d / kCluster > kMaxSlice || d % (kCluster * 4) != 0) {
    *msg = "model width d must be a multiple of 32 and at most 1280 for the block projections";
    return cudaErrorInvalidValue;
  }
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const size_t dec_bytes = decode_workspace_bytes(a.B, a.T, 1, a.H, 1);
  const size_t rows = align256(static_cast<size_t>(a.B) * d * sizeof(float));
  float* q = reinterpret_cast<float*>(ws + dec_bytes);
  float* att = reinterpret_cast<float*>(ws + dec_bytes + rows);
  if (fused_block_supported(a.H, 64)) {
    // up to 8 heads: LayerNorm, query, attention (and, when a cluster of H CTAs per
    // slot fits for every slot at once, the out projection too) in one kernel
    bool gathered = false;
    cudaError_t e = launch_block_fused(a, att, &gathered, dev, stream);
    if (e != cudaSuccess || gathered) return e;
    return launch_gemv<false>(att, nullptr, nullptr, 0.f, a.WO, a.bO, a.x, a.x, a.B, d, dev.device, stream);
  }

  // 1. h = LayerNorm(x); q = h x WQ + bQ
  cudaError_t e = launch_gemv<true>(a.x, a.gamma, a.beta, a.eps, a.WQ, a.bQ, nullptr, q, a.B, d, dev.device, stream);
  if (e != cudaSuccess) return e;
  // 2. attention of q over layer l's cache
  DecodeLaunch dl;
  dl.Kc = a.Kc;
  dl.Vc = a.Vc;
  dl.Q = q;
  dl.key_len = a.key_len;
  dl.out = att;
  dl.nq = 1;
  dl.l0 = a.layer;
  dl.nl = 1;
  dl.key_len_add = 0;
  dl.workspace = ws;
  dl.B = a.B;
  dl.T = a.T;
  dl.L = a.L;
  dl.H = a.H;
  dl.scale = a.scale;
  dl.cache_bf16 = a.cache_bf16;
  e = launch_decode(dl, dev, stream, msg);
  if (e != cudaSuccess) return e;
  // 3. x = x + a x WO + bO
  return launch_gemv<false>(att, nullptr, nullptr, 0.f, a.WO, a.bO, a.x, a.x, a.B, d, dev.device, stream);
}

}  // namespace cxa
