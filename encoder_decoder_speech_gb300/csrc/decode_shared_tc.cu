// Shared-cache multi-query decode on the tensor cores: nq (3..16) query rows per
// (slot, layer, head) attend the slot's one bf16 cache, the batch-N-over-one-
// shared-cache case of SharedSplitKVCached ("Caso de estudio: WhisperKit", §3).
//
// The work split, the segment flush and the last-arriver merge are those of the
// stream decode kernel (decode.cu). A 128-key chunk goes through two tcgen05
// products with fp32 accumulators in tensor memory:
//
//  * scores: S^T[128 keys x 16 queries] = K_chunk[128 x 64] Q^T (kind::f16,
//    both operands K-major, 128-byte swizzle). K arrives by TMA from a 3-D view
//    of the cache (c, t, slot*L*H + l*H + h); the Q tile (queries pre-scaled by
//    scale*log2(e), rounded to bf16, rows >= nq zero) is written by the MMA
//    warp at each row start. Double-buffered in TMEM.
//  * softmax on the CUDA cores: each of the 128 consumer threads owns one key
//    and reads its scores with one tcgen05.ld; the chunk max of a query is one
//    redux.sync per warp plus a 4-entry shared-memory max; probabilities are
//    written, rounded to bf16, as P^T[query][key] in the 128-byte-swizzled
//    K-major layout, and the running sums add the same rounded values so that
//    the weights of the final average sum to one exactly.
//  * values: O_chunk[128 x 64] = P^T[128 x 128 keys] V_chunk[128 x 64] with V
//    MN-major straight from its TMA tile (keys = K, channels = N). Only the
//    first 16 rows of the A operand are queries; the other 112 rows the MMA
//    reads fall on later shared memory and produce accumulator lanes nobody
//    reads, so the P buffer stays 4 KB. Double-buffered in TMEM.
//  * consumer warp 0, whose TMEM lanes hold the query rows, adds each chunk's
//    O into a running accumulator kept in TMEM (acc = acc * corr + O_chunk,
//    one chunk behind so that the P.V product overlaps the next softmax) and
//    writes the segment's result or partial slot at the row's end.
//
// V rows past the key length of a tail chunk are zeroed in shared memory before
// the product: their probabilities are 0 and stale rows may hold any bits.
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
constexpr int kChunk = 128;                    // keys per chunk: M of the scores, K of P.V
constexpr int kNPad = 16;                      // query columns of the score MMA (rows >= nq zero)
constexpr int kRowBytes = kDh * 2;             // one bf16 row of 64 channels
constexpr int kBoxRows = 32;                   // keys per TMA box
constexpr int kBoxBytes = kBoxRows * kRowBytes;
constexpr int kTileBytes = kChunk * kRowBytes; // K or V of one chunk: 16 KB
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kStages = 3;
constexpr int kPBytes = 4096;                  // P^T of a chunk: 2 key halves x 16 rows x 128 B
constexpr int kQTileBytes = kNPad * kRowBytes; // 2 KB
constexpr int kConsumerWarps = 4;              // one key per consumer thread
constexpr int kThreads = (kConsumerWarps + 2) * 32;   // + producer warp + MMA warp
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMmaWarp = kConsumerWarps + 1;
constexpr int kCtasPerSm = 2;
constexpr uint32_t kTmemCols = 256;            // S: 2 x 16 at 0, O: 2 x 64 at 64, acc: 64 at 192
constexpr uint32_t kOCol = 64;
constexpr uint32_t kAccCol = 192;
constexpr int kBars = 2 * kStages + 10;        // full, empty, tfull, tempty, pfull, ofull, oempty
// P buffers sit first: rows 16..127 of the P.V A operand read up to 16 KB past a
// buffer's key half, which must stay inside this CTA's shared memory.
constexpr int kPRegion = 2 * kPBytes;
static_assert(kPRegion + kStages * kStageBytes >= kPBytes + 2048 + 16 * 1024, "A-operand overread");

struct TcParams {
  const float* Q;
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
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
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

template <int kNQT>   // query columns the softmax handles (4, 8 or 16 >= nq)
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_shared_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                            const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  // layout: P^T x 2 | stages [K tile | V tile] x kStages | Q tiles x 2 | small arrays
  const uint32_t p_base = base;
  const uint32_t stage_base = base + kPRegion;
  const uint32_t q_base = stage_base + kStages * kStageBytes;
  float* s_red = reinterpret_cast<float*>(bp + kPRegion + kStages * kStageBytes + 2 * kQTileBytes);  // [4][16]
  float* s_fin = s_red + kConsumerWarps * kNPad;                      // [16] m, [16] S of the segment
  float* s_corr = s_fin + 2 * kNPad;                                  // [2][16] per-chunk rescale factors
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_corr + 2 * kNPad);
  long long* s_first = reinterpret_cast<long long*>(bars + kBars);
  int* s_nch = reinterpret_cast<int*>(s_first + p.B + 1);
  volatile int* s_flags = reinterpret_cast<volatile int*>(s_nch + p.B + (p.B & 1));   // abort, last, tmem base
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[kStages + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * kStages + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * kStages + 2 + a]); };
  auto pfull_bar = [&](int a) { return smem_u32(&bars[2 * kStages + 4 + a]); };
  auto ofull_bar = [&](int a) { return smem_u32(&bars[2 * kStages + 6 + a]); };
  auto oempty_bar = [&](int a) { return smem_u32(&bars[2 * kStages + 8 + a]); };

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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kConsumerWarps);
      mbar_init(pfull_bar(a), 1);
      mbar_init(ofull_bar(a), 1);
      mbar_init(oempty_bar(a), 1);
    }
    fence_mbar_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(const_cast<int*>(&s_flags[2])), kTmemCols);
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
      Cursor cur = locate(g0, s_first, s_nch, p.B);
      uint32_t armed = 0, armed_parity = 0;
      bool ok = true;
      for (long long g = g0, i = 0; g < g1; ++g, ++i) {
        const int s = static_cast<int>(i % kStages);
        const uint32_t parity = static_cast<uint32_t>((i / kStages) & 1);
        if (!mbar_wait(empty_bar(s), parity ^ 1u, s_flags)) {
          ok = false;
          break;
        }
        const int kl = min(max(__ldg(p.key_len + cur.b), 0), p.T);
        const int t0 = cur.c * kChunk;
        const int nbox = (min(kChunk, kl - t0) + kBoxRows - 1) / kBoxRows;   // rows past them stay stale
        const int crow = cur.b * p.LHc + p.lh0 + cur.lh;
        const uint32_t dst = stage_base + s * kStageBytes;
        mbar_arrive_expect_tx(full_bar(s), static_cast<uint32_t>(2 * nbox * kBoxBytes));
        for (int j = 0; j < nbox; ++j) {
          tma_load_3d(dst + j * kBoxBytes, &tmK, full_bar(s), 0, t0 + j * kBoxRows, crow);
          tma_load_3d(dst + kTileBytes + j * kBoxBytes, &tmV, full_bar(s), 0, t0 + j * kBoxRows, crow);
        }
        armed |= 1u << s;
        armed_parity = (armed_parity & ~(1u << s)) | (parity << s);
        advance(cur, s_nch, p.B, LH);
      }
      if (!ok) {
        s_flags[0] = 1;
        atomicOr(p.status, 1u);
        for (int s = 0; s < kStages; ++s)
          if (armed & (1u << s)) mbar_wait(full_bar(s), (armed_parity >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (active && warp == kMmaWarp) {
    // ------------------------------------------------------------ Q tiles + MMA issue
    constexpr uint32_t idesc_s = make_idesc(1u, kChunk, kNPad);
    constexpr uint32_t idesc_o = make_idesc(1u, 128, kDh) | (1u << 16);   // B (V) MN-major
    Cursor cur = locate(g0, s_first, s_nch, p.B);
    int qbuf = 1, prev_b = -1, prev_lh = -1;
    bool ok = true;
    // P.V of chunk j: A = P^T buffer j&1, B = V of its stage, D = O buffer j&1.
    auto issue_pv = [&](long long j) {
      const int b = static_cast<int>(j & 1);
      const uint32_t par = static_cast<uint32_t>((j >> 1) & 1);
      if (!mbar_wait(pfull_bar(b), par, s_flags) || !mbar_wait(oempty_bar(b), par ^ 1u, s_flags)) {
        ok = false;
        return;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t pt = p_base + b * kPBytes;
        const uint32_t vt = stage_base + static_cast<uint32_t>(j % kStages) * kStageBytes + kTileBytes;
        const uint32_t d_tmem = tmem_base + kOCol + static_cast<uint32_t>(b) * kDh;
#pragma unroll
        for (int kb = 0; kb < kChunk / 16; ++kb) {
          const uint64_t ad = smem_desc_k_sw128(pt + (kb >> 2) * 2048 + (kb & 3) * 32);
          const uint64_t bd = smem_desc_mn_sw128(vt + kb * 2048);
          mma_bf16(d_tmem, ad, bd, idesc_o, kb != 0 ? 1u : 0u);
        }
        tc_commit(ofull_bar(b));
        tc_commit(empty_bar(static_cast<int>(j % kStages)));
      }
      __syncwarp();
    };
    long long i = 0;
    for (long long g = g0; g < g1 && ok; ++g, ++i) {
      const int s = static_cast<int>(i % kStages);
      const uint32_t parity = static_cast<uint32_t>((i / kStages) & 1);
      const int acc = static_cast<int>(i & 1);
      const uint32_t acc_parity = static_cast<uint32_t>((i >> 1) & 1);
      if (!mbar_wait(tempty_bar(acc), acc_parity ^ 1u, s_flags)) {
        ok = false;
        break;
      }
      if (cur.b != prev_b || cur.lh != prev_lh) {
        // A new row: its queries become the B operand of the scores. The buffer was
        // last read by the MMAs of the row before the previous one, finished since
        // the consumers released the score accumulator just waited on.
        qbuf ^= 1;
        const uint32_t qt = q_base + qbuf * kQTileBytes;
        // 16 rows x 64 channels: lane handles row (lane / 2), half (lane & 1) of the channels
        const int qr = lane >> 1, half = lane & 1;
        const bool valid = qr < nq;
        const float* src = p.Q + qrow(cur.b, cur.lh, valid ? qr : 0) * kDh + half * 32;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float4 f = valid ? __ldg(reinterpret_cast<const float4*>(src) + 2 * j + k)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            __nv_bfloat162 lo = __floats2bfloat162_rn(f.x * p.qscale, f.y * p.qscale);
            __nv_bfloat162 hi = __floats2bfloat162_rn(f.z * p.qscale, f.w * p.qscale);
            w[2 * k] = *reinterpret_cast<uint32_t*>(&lo);
            w[2 * k + 1] = *reinterpret_cast<uint32_t*>(&hi);
          }
          // row qr: 128 bytes = 8 chunks of 8 bf16; this lane writes chunks 4*half .. 4*half+3
          const uint32_t chunk = static_cast<uint32_t>(4 * half + j);
          st_shared_v4(qt + qr * 128 + ((chunk ^ (qr & 7)) << 4), w[0], w[1], w[2], w[3]);
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
        const uint32_t kt = stage_base + s * kStageBytes;
        const uint32_t qt = q_base + qbuf * kQTileBytes;
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kNPad);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(d_tmem, smem_desc_k_sw128(kt + k * 32), smem_desc_k_sw128(qt + k * 32), idesc_s, k != 0 ? 1u : 0u);
        tc_commit(tfull_bar(acc));
      }
      __syncwarp();
      if (i > 0) issue_pv(i - 1);   // the previous chunk's P.V overlaps this chunk's softmax
      advance(cur, s_nch, p.B, LH);
    }
    if (ok && i > 0) issue_pv(i - 1);
    if (!ok) {
      s_flags[0] = 1;
      atomicOr(p.status, 1u);
    }
  } else if (active) {
    // ------------------------------------------------------------ consumers
    const int tid = threadIdx.x;                   // 0..127: key of the chunk for the softmax
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // P^T address of (query q, key tid) in buffer 0: key half, 8-row group, swizzled 16-byte chunk
    const int kk = tid & 63;
    const uint32_t p_key = static_cast<uint32_t>((tid >> 6) * 2048 + (kk & 7) * 2);
    const uint32_t p_chunk = static_cast<uint32_t>(kk >> 3);
    Cursor cur = locate(g0, s_first, s_nch, p.B);
    int seg_c0 = cur.c;
    float m_run[kNQT], s_run[kNQT];
#pragma unroll
    for (int q = 0; q < kNQT; ++q) {
      m_run[q] = -INFINITY;
      s_run[q] = 0.f;
    }
    bool ok = true, pending = false, acc_empty = true;
    auto fail = [&]() {
      ok = false;
      s_flags[0] = 1;
      atomicOr(p.status, 1u);
    };
    // Warp 0 only: acc = acc * corr_j + O_j in TMEM (lane q = query q). With final
    // set, lane q < nq writes mul * (acc * corr_j + O_j) to dst instead (16 channels
    // at a time; zeros after a failed wait).
    auto add_chunk = [&](long long j, bool final, float* dst, float mul) {
      const int b = static_cast<int>(j & 1);
      if (ok && !mbar_wait(ofull_bar(b), static_cast<uint32_t>((j >> 1) & 1), s_flags)) fail();
      tc_fence_after();
      const float corr = lane < kNPad ? s_corr[b * kNPad + lane] : 0.f;
#pragma unroll
      for (int h = 0; h < kDh / 16; ++h) {
        uint32_t o[16], acc[16];
        tmem_ld_32x32b_x16(tmem_base + kOCol + static_cast<uint32_t>(b * kDh + h * 16), o);
        if (!acc_empty) tmem_ld_32x32b_x16(tmem_base + kAccCol + static_cast<uint32_t>(h * 16), acc);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          acc[c] = __float_as_uint(acc_empty ? __uint_as_float(o[c])
                                             : fmaf(__uint_as_float(acc[c]), corr, __uint_as_float(o[c])));
        if (final) {
          if (lane < nq) {
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              *reinterpret_cast<float4*>(dst + h * 16 + c) =
                  ok ? make_float4(__uint_as_float(acc[c]) * mul, __uint_as_float(acc[c + 1]) * mul,
                                   __uint_as_float(acc[c + 2]) * mul, __uint_as_float(acc[c + 3]) * mul)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        } else {
          tmem_st_32x32b_x16(tmem_base + kAccCol + static_cast<uint32_t>(h * 16), acc);
        }
      }
      if (!final) tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(oempty_bar(b));
      acc_empty = final;
    };

    for (long long g = g0, i = 0; g < g1; ++g, ++i) {
      const int s = static_cast<int>(i % kStages);
      const int a = static_cast<int>(i & 1);
      const uint32_t acc_parity = static_cast<uint32_t>((i >> 1) & 1);
      const int kl = min(max(__ldg(p.key_len + cur.b), 0), p.T);
      const int nch = s_nch[cur.b];
      const int n = min(kChunk, kl - cur.c * kChunk);
      if (ok && !mbar_wait(tfull_bar(a), acc_parity, s_flags)) fail();
      tc_fence_after();
      uint32_t sr[16];
      tmem_ld_32x32b_x16(tmem_base + lane_base + static_cast<uint32_t>(a * kNPad), sr);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(a));

      // ---- softmax of the chunk: thread tid owns key tid
      const bool valid_key = tid < n && ok;
      float sc[kNQT];
#pragma unroll
      for (int q = 0; q < kNQT; ++q) {
        sc[q] = valid_key ? __uint_as_float(sr[q]) : -INFINITY;
        const float mq = warp_max(sc[q]);
        if (lane == 0) s_red[warp * kNPad + q] = mq;
      }
      named_barrier(1, kConsumerWarps * 32);
      const uint32_t pt = p_base + a * kPBytes + p_key;
#pragma unroll
      for (int q = 0; q < kNQT; ++q) {
        float M = m_run[q];
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, s_red[w * kNPad + q]);
        const float corr = M == -INFINITY ? 1.f : rescale(m_run[q], M);
        m_run[q] = M;
        const __nv_bfloat16 pb = __float2bfloat16_rn(valid_key ? exp2f(sc[q] - M) : 0.f);
        s_run[q] = s_run[q] * corr + __bfloat162float(pb);
        if (tid == 0) s_corr[a * kNPad + q] = corr;   // the same in every thread
        const int r = q & 7;
        st_shared_u16(pt + (q >> 3) * 1024 + r * 128 + ((p_chunk ^ static_cast<uint32_t>(r)) << 4),
                      __bfloat16_as_ushort(pb));
      }
      if (n < kChunk) {
        // tail chunk: zero the V rows of keys >= n (their P is 0; the rows may hold any bits)
        if (ok && !mbar_wait(full_bar(s), static_cast<uint32_t>((i / kStages) & 1), s_flags)) fail();
        const uint32_t vt = stage_base + s * kStageBytes + kTileBytes;
        for (int u = n * (kRowBytes / 16) + tid; u < kTileBytes / 16; u += kConsumerWarps * 32)
          st_shared_v4(vt + u * 16, 0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      named_barrier(1, kConsumerWarps * 32);                 // P^T (and the V tail) complete
      if (tid == 0) mbar_arrive(pfull_bar(a));
      if (warp == 0 && pending) add_chunk(i - 1, false, nullptr, 0.f);
      pending = true;

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
        named_barrier(1, kConsumerWarps * 32);
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
        if (warp == 0) {
          const int ql = lane < nq ? lane : nq - 1;
          const float S = s_fin[kNPad + ql];
          float* dst;
          float mul = 1.f;
          if (whole_row) {
            dst = p.out + qrow(cur.b, cur.lh, ql) * kDh;
            mul = S > 0.f ? 1.f / S : 0.f;
          } else {
            float* P = p.part + ((row * nq + ql) * p.part_stride + seg) * kPartFloats;
            if (lane < nq) {
              P[0] = ok ? s_fin[ql] : -INFINITY;
              P[1] = ok ? S : 0.f;
            }
            dst = P + 4;
          }
          add_chunk(i, true, dst, mul);
          pending = false;
        } else {
          pending = false;
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
    tmem_dealloc(tmem_base, kTmemCols);
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

size_t smem_bytes(int B) {
  size_t n = 1024 + kPRegion + static_cast<size_t>(kStages) * kStageBytes + 2 * kQTileBytes;
  n += (kConsumerWarps * kNPad + 4 * kNPad) * 4 + kBars * 8;
  n += static_cast<size_t>(B + 1) * 8 + static_cast<size_t>(B + (B & 1)) * 4 + 16;
  return n;
}

// A 3-D view (channel, t, slot*L*H + l*H + h) of a bf16 cache, 32-key boxes of
// one 128-byte row each, swizzled for the MMA.
bool encode_cache_map(EncodeTiledFn encode, CUtensorMap* map, const void* cache, const TcParams& prm,
                      const char* what, std::string* msg) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDh), static_cast<cuuint64_t>(prm.T),
                        static_cast<cuuint64_t>(prm.B) * prm.LHc};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes), static_cast<cuuint64_t>(prm.T) * kRowBytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kDh), kBoxRows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(cache), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *msg = std::string("cuTensorMapEncodeTiled failed for the ") + what + " cache (code " +
           std::to_string(static_cast<int>(r)) + ")";
    return false;
  }
  return true;
}

template <int kNQT>
cudaError_t launch_tc(const TcParams& prm, const void* Kc, const void* Vc, const DeviceInfo& dev,
                      cudaStream_t stream, std::string* msg) {
  EncodeTiledFn encode = encoder();
  if (encode == nullptr) {
    *msg = "cuTensorMapEncodeTiled is not available from the CUDA driver";
    return cudaErrorInvalidValue;
  }
  CUtensorMap tmK, tmV;
  if (!encode_cache_map(encode, &tmK, Kc, prm, "K", msg) || !encode_cache_map(encode, &tmV, Vc, prm, "V", msg))
    return cudaErrorInvalidValue;
  static std::mutex mu;
  static size_t attr_bytes[128] = {};
  const size_t smem = smem_bytes(prm.B);
  {
    std::lock_guard<std::mutex> lock(mu);
    const int d = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
    if (attr_bytes[d] < smem) {
      cudaError_t e = cudaFuncSetAttribute(decode_shared_tc_kernel<kNQT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      // two CTAs per SM need the largest shared-memory carveout
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_shared_tc_kernel<kNQT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      attr_bytes[d] = smem;
    }
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_shared_tc_kernel<kNQT>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  if (per_sm < kCtasPerSm) {
    // The occupancy query reports one CTA per SM for kernels that allocate tensor
    // memory. Two of these fit by registers, shared memory and TMEM columns
    // (2 x 256 of 512), and no CTA waits on another, so the count is taken from
    // the register and shared-memory budgets instead.
    static int fits[128] = {};
    const int d = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
    if (fits[d] == 0) {
      cudaFuncAttributes fa;
      cudaDeviceProp pr;
      e = cudaFuncGetAttributes(&fa, decode_shared_tc_kernel<kNQT>);
      if (e == cudaSuccess) e = cudaGetDeviceProperties(&pr, dev.device);
      if (e != cudaSuccess) return e;
      const long long regs_cta = static_cast<long long>((fa.numRegs + 7) / 8 * 8) * kThreads;
      const long long smem_cta = static_cast<long long>(smem + fa.sharedSizeBytes + pr.reservedSharedMemPerBlock);
      const bool two = 2 * regs_cta <= pr.regsPerMultiprocessor &&
                       2 * smem_cta <= static_cast<long long>(pr.sharedMemPerMultiprocessor) &&
                       2 * kThreads <= pr.maxThreadsPerMultiProcessor;
      fits[d] = two ? 2 : 1;
    }
    if (fits[d] > per_sm) per_sm = fits[d];
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dev.num_sms * (per_sm < kCtasPerSm ? per_sm : kCtasPerSm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_shared_tc_kernel<kNQT>, tmK, tmV, prm);
}

size_t counters_bytes(int B, int L, int H) {
  const size_t n = static_cast<size_t>(B) * L * H * sizeof(unsigned int);
  return (n + 255) & ~static_cast<size_t>(255);
}

}  // namespace

cudaError_t launch_decode_shared_tc(const DecodeLaunch& a, const DeviceInfo& dev, cudaStream_t stream,
                                    std::string* msg) {
  if (!a.cache_bf16) {
    *msg = "the tensor-core shared decode serves bf16 caches";
    return cudaErrorInvalidValue;
  }
  TcParams prm;
  prm.Q = a.Q;
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
  cudaError_t e = a.nq <= 4   ? launch_tc<4>(prm, a.Kc, a.Vc, dev, stream, msg)
                  : a.nq <= 8 ? launch_tc<8>(prm, a.Kc, a.Vc, dev, stream, msg)
                              : launch_tc<16>(prm, a.Kc, a.Vc, dev, stream, msg);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace cxa
