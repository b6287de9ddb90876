// Shared-cache multi-query decode with tensor-core scores: nq (3..16) query rows
// per (slot, layer, head) attend the slot's one cache, the batch-N-over-one-
// shared-cache case of SharedSplitKVCached ("Caso de estudio: WhisperKit", §3).
//
// The work split, the producer ring, the segment flush and the last-arriver
// merge are those of the stream decode kernel (decode.cu). What changes is the
// arithmetic of a 128-key chunk:
//
//  * scores on tcgen05: S^T[128 keys x 16 queries] = K_chunk[128 x 64] Q^T,
//    kind::f16 (bf16 cache, queries rounded to bf16; the kernel is written for
//    kind::tf32 too, but an fp32 cache keeps the fp32 CUDA-core scores of
//    decode.cu, whose error bar TF32 operands would not meet). Both
//    operands are K-major with 128-byte swizzling: the K tile arrives by TMA
//    from a 3-D view of the cache (c, t, slot*L*H + l*H + h), the Q tile
//    (queries pre-scaled by scale*log2(e), rows >= nq zero) is written into
//    shared memory by the MMA warp at each row start (double-buffered). The
//    accumulator (16 fp32 columns) is double-buffered in TMEM.
//  * softmax: each of the 128 consumer threads owns one key and reads its 16
//    scores with one tcgen05.ld; per query, the chunk max is a warp + shared
//    memory reduction, each probability is one exp2 and each thread keeps its
//    own running sums (rescaled by the common running max).
//  * P.V on the CUDA cores: thread (channel pair, query quad) owns 8 output
//    accumulators and walks the chunk's keys: P rows from shared memory, V rows
//    from the stage (bulk-copied, valid keys only).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace cxa {
namespace {

constexpr int kDh = 64;
constexpr int kPartFloats = 68;
constexpr int kPartChunk = 64;
constexpr int kChunk = 128;                 // keys per chunk = MMA M
constexpr int kNPad = 16;                   // queries per MMA (N), rows >= nq are zero
constexpr int kConsumerWarps = 4;           // one key per consumer thread
constexpr int kThreads = (kConsumerWarps + 2) * 32;   // + producer warp + MMA warp
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMmaWarp = kConsumerWarps + 1;
constexpr int kPStride = kNPad + 4;         // floats per key row of P in shared memory (padded)

template <bool kBF16>
struct TcTraits {
  static constexpr int kElem = kBF16 ? 2 : 4;
  static constexpr int kRowBytes = kDh * kElem;              // 128 / 256
  static constexpr int kKHalves = kRowBytes / 128;           // 128-byte column blocks of a K row: 1 / 2
  static constexpr int kKTileBytes = kChunk * kRowBytes;     // 16 / 32 KB (swizzled, kKHalves boxes)
  static constexpr int kVBytes = kChunk * kRowBytes;         // 16 / 32 KB (plain rows)
  static constexpr int kStageBytes = kKTileBytes + kVBytes;
  static constexpr int kStages = 2;
  static constexpr int kQTileBytes = kNPad * kRowBytes;      // 2 / 4 KB per Q buffer (swizzled)
  static constexpr int kMmaK = kBF16 ? 16 : 8;               // K of one MMA
  static constexpr int kMmasPer128B = 128 / (kMmaK * kElem); // 4
  static constexpr int kCtasPerSm = kBF16 ? 2 : 1;
};

struct TcParams {
  const float* Q;
  const uint8_t* Vc;
  const int* key_len;
  float* out;
  float* part;
  unsigned int* counters;
  unsigned int* status;
  int B, T, LH, LHc, lh0, nq, part_stride;
  float qscale;
};

__device__ __forceinline__ float rescale(float m, float M) { return m == -INFINITY ? 0.f : exp2f(m - M); }
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

struct Cursor {
  int b, lh, c;
};
__device__ __forceinline__ Cursor locate(long long g, const long long* s_first, const int* s_nch, int B) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_first[mid] <= g) lo = mid; else hi = mid - 1;
  }
  const long long local = g - s_first[lo];
  Cursor cur;
  cur.b = lo;
  cur.lh = static_cast<int>(local / s_nch[lo]);
  cur.c = static_cast<int>(local - static_cast<long long>(cur.lh) * s_nch[lo]);
  return cur;
}
__device__ __forceinline__ void advance(Cursor& cur, const int* s_nch, int B, int LH) {
  if (++cur.c < s_nch[cur.b]) return;
  cur.c = 0;
  if (++cur.lh < LH) return;
  cur.lh = 0;
  do {
    ++cur.b;
  } while (cur.b < B && s_nch[cur.b] == 0);
}
__device__ __forceinline__ long long owner_of(long long g, long long total, long long ranges) {
  return ((g + 1) * ranges + total - 1) / total - 1;
}

template <bool kBF16, int kNQT>   // kNQT = query columns the softmax handles (4, 8 or 16 >= nq)
__global__ void __launch_bounds__(kThreads, TcTraits<kBF16>::kCtasPerSm)
    decode_shared_tc_kernel(const __grid_constant__ CUtensorMap tmK, const TcParams p) {
  using R = TcTraits<kBF16>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  // layout: stages [K tile | V rows] x kStages, Q tiles x 2, P [128][kPStride] f32, then small arrays
  uint8_t* stage_ptr = bp;
  uint8_t* qtile_ptr = bp + R::kStages * R::kStageBytes;
  float* sP = reinterpret_cast<float*>(qtile_ptr + 2 * R::kQTileBytes);
  float* s_red = sP + kChunk * kPStride;                           // [4 warps][16]
  float* s_fin = s_red + kConsumerWarps * kNPad;                   // [16] merged m, [16] merged s
  float* s_corr = s_fin + 2 * kNPad;                               // [16] this chunk's rescale factors
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_corr + 2 * kNPad); // full[S], empty[S], tfull[2], tempty[2]
  long long* s_first = reinterpret_cast<long long*>(bars + 2 * R::kStages + 4);
  int* s_nch = reinterpret_cast<int*>(s_first + p.B + 1);
  volatile int* s_flags = reinterpret_cast<volatile int*>(s_nch + p.B + (p.B & 1));   // abort, last, tmem base
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[R::kStages + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * R::kStages + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * R::kStages + 2 + a]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int LH = p.LH, nq = p.nq;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {   // chunk numbering from key_len (every CTA computes the same prefix)
    long long run = 0;
    for (int base_b = 0; base_b < p.B; base_b += 32) {
      const int b = base_b + lane;
      int nch = 0;
      if (b < p.B) {
        const int kl = min(max(__ldg(p.key_len + b), 0), p.T);
        nch = (kl + kChunk - 1) / kChunk;
        s_nch[b] = nch;
      }
      long long v = static_cast<long long>(nch) * LH;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
      }
      if (b < p.B) s_first[b] = run + v - static_cast<long long>(nch) * LH;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) {
      s_first[p.B] = run;
      s_flags[0] = 0;
      s_flags[1] = 0;
    }
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < R::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kConsumerWarps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kConsumerWarps);
    }
    fence_mbar_init();
    prefetch_tmap(&tmK);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(const_cast<int*>(&s_flags[2])), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = static_cast<uint32_t>(s_flags[2]);

  const long long total = s_first[p.B];
  const long long ranges = total < gridDim.x ? total : static_cast<long long>(gridDim.x);
  const bool active = total > 0 && blockIdx.x < ranges;
  const long long g0 = active ? blockIdx.x * total / ranges : 0;
  const long long g1 = active ? (blockIdx.x + 1) * total / ranges : 0;
  auto qrow = [&](int b, int lh, int n) { return (static_cast<long long>(b) * nq + n) * LH + lh; };

  // Q, out and the workspace may belong to the previous grid.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  {
    const long long per_slot = static_cast<long long>(nq) * LH * (kDh / 4);
    for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < p.B * per_slot;
         i += static_cast<long long>(gridDim.x) * kThreads)
      if (s_nch[static_cast<int>(i / per_slot)] == 0)
        reinterpret_cast<float4*>(p.out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  if (active && warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      Cursor cur = locate(g0, s_first, s_nch, p.B);
      uint32_t armed = 0, armed_parity = 0;
      bool ok = true;
      for (long long g = g0, i = 0; g < g1; ++g, ++i) {
        const int s = static_cast<int>(i % R::kStages);
        const uint32_t parity = static_cast<uint32_t>((i / R::kStages) & 1);
        if (!mbar_wait(empty_bar(s), parity ^ 1u, s_flags)) {
          ok = false;
          break;
        }
        const int kl = min(max(__ldg(p.key_len + cur.b), 0), p.T);
        const int t0 = cur.c * kChunk;
        const int n = min(kChunk, kl - t0);
        const int crow = cur.b * p.LHc + p.lh0 + cur.lh;
        const uint32_t kv_bytes = static_cast<uint32_t>(n) * R::kRowBytes;
        const uint32_t dst = smem_u32(stage_ptr + s * R::kStageBytes);
        mbar_arrive_expect_tx(full_bar(s), R::kKTileBytes + kv_bytes);
#pragma unroll
        for (int kh = 0; kh < R::kKHalves; ++kh)
          tma_load_3d(dst + kh * (kChunk * 128), &tmK, full_bar(s), kh * (128 / R::kElem), t0, crow);
        bulk_g2s_hint(dst + R::kKTileBytes, p.Vc + (static_cast<size_t>(crow) * p.T + t0) * R::kRowBytes, kv_bytes,
                      full_bar(s), pol);
        armed |= 1u << s;
        armed_parity = (armed_parity & ~(1u << s)) | (parity << s);
        advance(cur, s_nch, p.B, LH);
      }
      if (!ok) {
        s_flags[0] = 1;
        atomicOr(p.status, 1u);
        for (int s = 0; s < R::kStages; ++s)
          if (armed & (1u << s)) mbar_wait(full_bar(s), (armed_parity >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (active && warp == kMmaWarp) {
    // ------------------------------------------------------------ Q tiles + MMA issue
    constexpr uint32_t idesc = make_idesc(kBF16 ? 1u : 2u, kChunk, kNPad);
    Cursor cur = locate(g0, s_first, s_nch, p.B);
    int qbuf = 1, prev_b = -1, prev_lh = -1;
    bool ok = true;
    for (long long g = g0, i = 0; g < g1 && ok; ++g, ++i) {
      const int s = static_cast<int>(i % R::kStages);
      const uint32_t parity = static_cast<uint32_t>((i / R::kStages) & 1);
      const int acc = static_cast<int>(i & 1);
      const uint32_t acc_parity = static_cast<uint32_t>((i >> 1) & 1);
      if (!mbar_wait(tempty_bar(acc), acc_parity ^ 1u, s_flags)) {
        ok = false;
        break;
      }
      if (cur.b != prev_b || cur.lh != prev_lh) {
        // A new row: its queries become the B operand. The buffer was last read by
        // the MMAs of the row before the previous one, finished since the consumers
        // released the accumulator just waited on.
        qbuf ^= 1;
        const uint32_t qt = smem_u32(qtile_ptr + qbuf * R::kQTileBytes);
        // 16 rows x (64 channels): lane handles row (lane / 2), half (lane & 1) of the channels
        const int qr = lane >> 1, half = lane & 1;
        const bool valid = qr < nq;
        const float* src = p.Q + qrow(cur.b, cur.lh, valid ? qr : 0) * kDh + half * 32;
        float v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 f = valid ? __ldg(reinterpret_cast<const float4*>(src) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[4 * j] = f.x * p.qscale;
          v[4 * j + 1] = f.y * p.qscale;
          v[4 * j + 2] = f.z * p.qscale;
          v[4 * j + 3] = f.w * p.qscale;
        }
        if constexpr (kBF16) {
          // row qr: 128 bytes = 8 chunks of 8 bf16; this lane writes chunks 4*half .. 4*half+3
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              __nv_bfloat162 pr = __floats2bfloat162_rn(v[8 * j + 2 * k], v[8 * j + 2 * k + 1]);
              w[k] = *reinterpret_cast<uint32_t*>(&pr);
            }
            const uint32_t chunk = static_cast<uint32_t>(4 * half + j);
            st_shared_v4(qt + qr * 128 + ((chunk ^ (qr & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
        } else {
          // fp32 rows are two 128-byte halves (channels 0-31, 32-63), each a swizzled [16 x 128 B] block
          const uint32_t blk = qt + static_cast<uint32_t>(half) * (kNPad * 128);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(blk + qr * 128 + ((static_cast<uint32_t>(j) ^ (qr & 7)) << 4), __float_as_uint(v[4 * j]),
                         __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        prev_b = cur.b;
        prev_lh = cur.lh;
      }
      if (!mbar_wait(full_bar(s), parity, s_flags)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t kt = smem_u32(stage_ptr + s * R::kStageBytes);
        const uint32_t qt = smem_u32(qtile_ptr + qbuf * R::kQTileBytes);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kNPad);
#pragma unroll
        for (int kh = 0; kh < R::kKHalves; ++kh)
#pragma unroll
          for (int k = 0; k < R::kMmasPer128B; ++k) {
            const uint64_t ad = smem_desc_k_sw128(kt + kh * (kChunk * 128) + k * 32);
            const uint64_t bd = smem_desc_k_sw128(qt + kh * (kNPad * 128) + k * 32);
            const uint32_t accumulate = (kh | k) != 0 ? 1u : 0u;
            if constexpr (kBF16)
              mma_bf16(d_tmem, ad, bd, idesc, accumulate);
            else
              mma_tf32(d_tmem, ad, bd, idesc, accumulate);
          }
        tc_commit(tfull_bar(acc));
      }
      __syncwarp();
      advance(cur, s_nch, p.B, LH);
    }
    if (!ok) {
      s_flags[0] = 1;
      atomicOr(p.status, 1u);
    }
  } else if (active) {
    // ------------------------------------------------------------ consumers
    const int tid = threadIdx.x;                   // 0..127: key of the chunk for the softmax
    // P.V: lane = channel pair 2cp, 2cp+1; warp = (query quad qg, key slice ks).
    // With fewer than four query quads the chunk's keys are split between warps,
    // so every warp works; the slices' accumulators are added at the flush.
    const int cp = lane;
    const int nquads = (nq + 3) / 4;
    const int ksplit = nquads == 1 ? 4 : (nquads == 2 ? 2 : 1);
    const int qg = warp / ksplit;                  // queries 4qg .. 4qg+3
    const int ks = warp % ksplit;                  // keys [ks, ks+1) * kChunk / ksplit
    const int pv_queries = qg < nquads ? min(4, nq - 4 * qg) : 0;
    Cursor cur = locate(g0, s_first, s_nch, p.B);
    int seg_c0 = cur.c;
    float m_run[kNQT], s_run[kNQT], acc[4][2];
#pragma unroll
    for (int q = 0; q < kNQT; ++q) {
      m_run[q] = -INFINITY;
      s_run[q] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = 0.f;
    bool ok = true;

    for (long long g = g0, i = 0; g < g1; ++g, ++i) {
      const int s = static_cast<int>(i % R::kStages);
      const uint32_t parity = static_cast<uint32_t>((i / R::kStages) & 1);
      const int a = static_cast<int>(i & 1);
      const uint32_t acc_parity = static_cast<uint32_t>((i >> 1) & 1);
      const int kl = min(max(__ldg(p.key_len + cur.b), 0), p.T);
      const int nch = s_nch[cur.b];
      const int n = min(kChunk, kl - cur.c * kChunk);
      if (ok && !mbar_wait(tfull_bar(a), acc_parity, s_flags)) {
        ok = false;
        s_flags[0] = 1;
        atomicOr(p.status, 1u);
      }
      tc_fence_after();
      uint32_t sr[16];
      tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(a * kNPad), sr);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(a));

      // ---- softmax of the chunk: thread tid owns key tid
      const bool valid_key = tid < n && ok;
      float sc[kNQT];
#pragma unroll
      for (int q = 0; q < kNQT; ++q) sc[q] = valid_key ? __uint_as_float(sr[q]) : -INFINITY;
#pragma unroll
      for (int q = 0; q < kNQT; ++q) {
        float mq = sc[q];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, off));
        if (lane == 0) s_red[warp * kNPad + q] = mq;
      }
      named_barrier(1, kConsumerWarps * 32);
      float corr[kNQT];
#pragma unroll
      for (int q = 0; q < kNQT; ++q) {
        float M = m_run[q];
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, s_red[w * kNPad + q]);
        corr[q] = M == -INFINITY ? 1.f : rescale(m_run[q], M);
        m_run[q] = M;
        const float pw = valid_key ? exp2f(sc[q] - M) : 0.f;
        s_run[q] = s_run[q] * corr[q] + pw;
        sc[q] = pw;
      }
      if (tid == 0) {   // the rescale factors are the same in every thread
#pragma unroll
        for (int q = 0; q < kNQT; ++q) s_corr[q] = corr[q];
      }
#pragma unroll
      for (int q4 = 0; q4 < kNQT / 4; ++q4)
        *reinterpret_cast<float4*>(sP + tid * kPStride + 4 * q4) =
            make_float4(sc[4 * q4], sc[4 * q4 + 1], sc[4 * q4 + 2], sc[4 * q4 + 3]);
      if (ok && !mbar_wait(full_bar(s), parity, s_flags)) {   // V rows of this stage
        ok = false;
        s_flags[0] = 1;
        atomicOr(p.status, 1u);
      }
      named_barrier(1, kConsumerWarps * 32);                 // P complete

      // ---- P.V: thread (cp, qg): channels 2cp, 2cp+1 of queries 4qg .. 4qg+3
      if (pv_queries > 0 && ok) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float cj = s_corr[4 * qg + j];
          acc[j][0] *= cj;
          acc[j][1] *= cj;
        }
        const uint8_t* vrow = stage_ptr + s * R::kStageBytes + R::kKTileBytes;
        const int k_lo = ks * (kChunk / ksplit);
        const int k_hi = min(n, k_lo + kChunk / ksplit);
#pragma unroll 4
        for (int k = k_lo; k < k_hi; ++k) {
          float v0, v1;
          if constexpr (kBF16) {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(vrow + k * R::kRowBytes + cp * 4);
            v0 = __uint_as_float(u << 16);
            v1 = __uint_as_float(u & 0xFFFF0000u);
          } else {
            const float2 f = *reinterpret_cast<const float2*>(vrow + k * R::kRowBytes + cp * 8);
            v0 = f.x;
            v1 = f.y;
          }
          const float4 pk = *reinterpret_cast<const float4*>(sP + k * kPStride + 4 * qg);
          acc[0][0] = fmaf(pk.x, v0, acc[0][0]);
          acc[0][1] = fmaf(pk.x, v1, acc[0][1]);
          acc[1][0] = fmaf(pk.y, v0, acc[1][0]);
          acc[1][1] = fmaf(pk.y, v1, acc[1][1]);
          acc[2][0] = fmaf(pk.z, v0, acc[2][0]);
          acc[2][1] = fmaf(pk.z, v1, acc[2][1]);
          acc[3][0] = fmaf(pk.w, v0, acc[3][0]);
          acc[3][1] = fmaf(pk.w, v1, acc[3][1]);
        }
      }
      named_barrier(1, kConsumerWarps * 32);                 // P and the stage read by everyone
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));

      const bool row_ends = (cur.c == nch - 1) || (g + 1 == g1);
      if (row_ends) {
        // ---- sums over the keys (threads) per query
#pragma unroll
        for (int q = 0; q < kNQT; ++q) {
          float sq = s_run[q];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
          if (lane == 0) s_red[warp * kNPad + q] = sq;
        }
        named_barrier(1, kConsumerWarps * 32);
        if (tid < kNQT) {
          float S = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) S += s_red[w * kNPad + tid];
          s_fin[kNPad + tid] = S;
        }
        if (tid == 0) {   // the running maxima are the same in every thread
#pragma unroll
          for (int q = 0; q < kNQT; ++q) s_fin[q] = m_run[q];
        }
        // add the key slices' accumulators (sP is free: the next chunk rewrites it after a barrier)
        if (ksplit > 1) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float2*>(sP + (warp * 4 + j) * kDh + 2 * cp) = make_float2(acc[j][0], acc[j][1]);
        }
        named_barrier(1, kConsumerWarps * 32);
        if (ksplit > 1 && ks == 0) {
          for (int k2 = 1; k2 < ksplit; ++k2)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 o = *reinterpret_cast<const float2*>(sP + ((warp + k2) * 4 + j) * kDh + 2 * cp);
              acc[j][0] += o.x;
              acc[j][1] += o.y;
            }
        }
        const bool writer = ks == 0;                 // one warp per query quad writes
        const long long row = static_cast<long long>(cur.b) * LH + cur.lh;
        const bool whole_row = seg_c0 == 0 && cur.c == nch - 1;
        long long first_owner = 0;
        int nseg = 1, seg = 0;
        if (!whole_row) {
          const long long grow = s_first[cur.b] + static_cast<long long>(cur.lh) * nch;
          first_owner = owner_of(grow, total, ranges);
          nseg = static_cast<int>(owner_of(grow + nch - 1, total, ranges) - first_owner + 1);
          seg = static_cast<int>(blockIdx.x - first_owner);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j >= pv_queries || !writer) continue;
          const int q = 4 * qg + j;
          const float S = s_fin[kNPad + q];
          if (whole_row) {
            if (ok)
              *reinterpret_cast<float2*>(p.out + qrow(cur.b, cur.lh, q) * kDh + 2 * cp) =
                  make_float2(S > 0.f ? acc[j][0] / S : 0.f, S > 0.f ? acc[j][1] / S : 0.f);
          } else {
            float* P = p.part + ((row * nq + q) * p.part_stride + seg) * kPartFloats;
            *reinterpret_cast<float2*>(P + 4 + 2 * cp) = make_float2(ok ? acc[j][0] : 0.f, ok ? acc[j][1] : 0.f);
            if (cp == 0) {
              P[0] = ok ? s_fin[q] : -INFINITY;
              P[1] = ok ? S : 0.f;
            }
          }
        }
        if (!whole_row) {
          __threadfence();
          named_barrier(1, kConsumerWarps * 32);
          if (tid == 0) {
            const unsigned int prev = atomicAdd(p.counters + row, 1u);
            s_flags[1] = (prev == static_cast<unsigned int>(nseg - 1)) ? 1 : 0;
          }
          named_barrier(1, kConsumerWarps * 32);
          if (s_flags[1]) {
            __threadfence();
            if (tid < kDh) {
              for (int q = 0; q < nq; ++q) {
                const float* P0 = p.part + (row * nq + q) * p.part_stride * kPartFloats;
                float MM = -INFINITY, SS = 0.f, AA = 0.f;
                for (int k = 0; k < nseg; ++k) {
                  const float mk = __ldcg(P0 + k * kPartFloats);
                  const float sk = __ldcg(P0 + k * kPartFloats + 1);
                  const float ak = __ldcg(P0 + k * kPartFloats + 4 + tid);
                  const float M2 = fmaxf(MM, mk);
                  const float f0 = rescale(MM, M2), f1 = rescale(mk, M2);
                  SS = SS * f0 + sk * f1;
                  AA = AA * f0 + ak * f1;
                  MM = M2;
                }
                p.out[qrow(cur.b, cur.lh, q) * kDh + tid] = SS > 0.f ? AA / SS : 0.f;
              }
            }
            if (tid == 0) p.counters[row] = 0u;
          }
        }
        named_barrier(1, kConsumerWarps * 32);
#pragma unroll
        for (int q = 0; q < kNQT; ++q) {
          m_run[q] = -INFINITY;
          s_run[q] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = 0.f;
      }
      const int pb = cur.b, plh = cur.lh;
      advance(cur, s_nch, p.B, LH);
      if (cur.b != pb || cur.lh != plh) seg_c0 = cur.c;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

template <bool kBF16>
size_t smem_bytes(int B) {
  using R = TcTraits<kBF16>;
  size_t n = 1024 + static_cast<size_t>(R::kStages) * R::kStageBytes + 2 * R::kQTileBytes;
  n += static_cast<size_t>(kChunk) * kPStride * 4 + (kConsumerWarps * kNPad + 4 * kNPad) * 4;
  n += (2 * R::kStages + 4) * 8 + static_cast<size_t>(B + 1) * 8 + static_cast<size_t>(B + (B & 1)) * 4 + 16;
  return n;
}

template <bool kBF16, int kNQT>
cudaError_t launch_tc(const TcParams& prm, const void* Kc, const DeviceInfo& dev, cudaStream_t stream,
                      std::string* msg) {
  using R = TcTraits<kBF16>;
  EncodeTiledFn encode = encoder();
  if (encode == nullptr) {
    *msg = "cuTensorMapEncodeTiled is not available from the CUDA driver";
    return cudaErrorInvalidValue;
  }
  CUtensorMap tmK;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(prm.T), static_cast<cuuint64_t>(prm.B) * prm.LHc};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(R::kRowBytes), static_cast<cuuint64_t>(prm.T) * R::kRowBytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / R::kElem), kChunk, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(&tmK, kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                      const_cast<void*>(Kc), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *msg = "cuTensorMapEncodeTiled failed for the K cache (code " + std::to_string(static_cast<int>(r)) + ")";
    return cudaErrorInvalidValue;
  }
  static std::mutex mu;
  static size_t attr_bytes[128] = {};
  const size_t smem = smem_bytes<kBF16>(prm.B);
  {
    std::lock_guard<std::mutex> lock(mu);
    const int d = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
    if (attr_bytes[d] < smem) {
      cudaError_t e = cudaFuncSetAttribute(decode_shared_tc_kernel<kBF16, kNQT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_bytes[d] = smem;
    }
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_shared_tc_kernel<kBF16, kNQT>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dev.num_sms * (per_sm < R::kCtasPerSm ? per_sm : R::kCtasPerSm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_shared_tc_kernel<kBF16, kNQT>, tmK, prm);
}

size_t counters_bytes(int B, int L, int H) {
  const size_t n = static_cast<size_t>(B) * L * H * sizeof(unsigned int);
  return (n + 255) & ~static_cast<size_t>(255);
}

}  // namespace

cudaError_t launch_decode_shared_tc(const DecodeLaunch& a, const DeviceInfo& dev, cudaStream_t stream,
                                    std::string* msg) {
  TcParams prm;
  prm.Q = a.Q;
  prm.Vc = static_cast<const uint8_t*>(a.Vc);
  prm.key_len = a.key_len;
  prm.out = a.out;
  prm.counters = static_cast<unsigned int*>(a.workspace);
  prm.part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + counters_bytes(a.B, a.nl, a.H));
  prm.status = dev.status_word;
  prm.B = a.B;
  prm.T = a.T;
  prm.LH = a.nl * a.H;
  prm.LHc = a.L * a.H;
  prm.lh0 = a.l0 * a.H;
  prm.nq = a.nq;
  prm.part_stride = (a.T + kPartChunk - 1) / kPartChunk;
  prm.qscale = a.scale * 1.4426950408889634f;
  if (!a.cache_bf16) {
    *msg = "the tensor-core shared decode serves bf16 caches";
    return cudaErrorInvalidValue;
  }
  cudaError_t e = a.nq <= 4   ? launch_tc<true, 4>(prm, a.Kc, dev, stream, msg)
                  : a.nq <= 8 ? launch_tc<true, 8>(prm, a.Kc, dev, stream, msg)
                              : launch_tc<true, 16>(prm, a.Kc, dev, stream, msg);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace cxa
