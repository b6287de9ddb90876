// Shared-cache multi-query decode on the tensor cores: nq (2..16) query rows per
// (slot, layer, head) attend the slot's one bf16 cache, the batch-N-over-one-
// shared-cache case of SharedSplitKVCached ("Caso de estudio: WhisperKit", §3).
//
// The work split and the segment flush are those of the stream decode kernel
// (decode.cu). A row cut by a range boundary leaves one partial state per CTA that
// works on it, and no CTA publishes a partial state (device fence, arrival
// counter) or merges a row while its K/V stream is running: with eight or more
// query columns a second, small kernel (decode_shared_merge_kernel, chained by
// programmatic dependent launch) merges the cut rows after the grid; with four
// (two to four queries), each CTA publishes its (at most two) cut rows at the end of its range and the
// last arriver of a row merges it. A 128-key chunk goes through two tcgen05
// products with fp32 accumulators in tensor memory:
//
//  * scores: S^T[128 keys x 32] = K_chunk[128 x 64] [Q_hi; Q_lo]^T (kind::f16,
//    both operands K-major, 128-byte swizzle). K arrives by TMA from a 3-D view
//    of the cache (c, t, slot*L*H + l*H + h); the queries, pre-scaled by
//    scale*log2(e), are split into bf16 hi and lo parts (rows >= nq zero) by the
//    MMA warp at each row start, so that a score is K.Q_hi + K.Q_lo with Q
//    carried to about 16 mantissa bits (K is exact: the cache is bf16).
//    Double-buffered in TMEM.
//  * softmax on the CUDA cores: each of the 128 consumer threads owns one key
//    and reads its scores with two tcgen05.ld (the hi and lo columns). Probabilities are taken against
//    a per-query reference max that moves only when some score passes it by
//    more than 2^8 (one bar.red.or per chunk tells); a move costs a warp
//    redux.sync and a 4-entry shared-memory max, plus, inside a row segment, a
//    rescale of the O accumulator in TMEM before the chunk's P.V is issued.
//    The MMA warp only builds Q tiles and issues the score MMAs; K and V stream
//    through separate rings of six tiles in all (a K stage returns once its score
//    MMA has run; two K and four V stages, three and three at sixteen columns).
//    Probabilities (<= 256) are written, rounded to bf16, as P[key][query]: one
//    32-byte row per key, eight queries to a 16-byte store, the row's two chunks
//    swapped every four keys (the 32-byte swizzle of an MN-major operand); the
//    running sums add the same rounded values, so the weights of the final
//    average sum to one exactly.
//  * values: O^T[64 channels x 16 queries] += V_chunk^T[64 x 128 keys] P[128 x 16]
//    (M = 64, N = 16): A is V MN-major straight from its TMA tile, B is P^T read
//    MN-major from P as written, accumulated over the row segment's chunks in TMEM (two
//    buffers, alternate segments). With M = 64 the accumulator rows sit in
//    lanes 0..15 of each warp's 32-lane quarter: channel 16w + l in lane
//    32w + l. A dedicated warp issues the chunk's P.V once the barrier that
//    completes P^T has let one consumer thread arrive on its mbarrier (and the
//    V tile has landed); an O rescale (rare) waits for the previous P.V's
//    commit and runs before it.
//  * at the end of a segment each consumer warp reads its 16 channels of O^T
//    and writes them for every query (result or the segment's partial slot).
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
#include "chunk_stream.cuh"
#include "ptx.cuh"

namespace cxa {
namespace {

constexpr int kDh = 64;
constexpr int kPartFloats = 68;
constexpr int kPartChunk = 64;
constexpr int kChunk = 128;                    // keys per chunk: M of the scores, K of P.V
constexpr int kNPad = 16;                      // query rows (>= nq zero)
constexpr int kSCols = 2 * kNPad;              // score MMA N: hi rows 0..15, lo rows 16..31 of Q
constexpr int kRowBytes = kDh * 2;             // one bf16 row of 64 channels
constexpr int kBoxRows = 32;                   // keys per TMA box
constexpr int kBoxBytes = kBoxRows * kRowBytes;
constexpr int kTileBytes = kChunk * kRowBytes; // K or V of one chunk: 16 KB
// K and V stream through separate rings sharing six 16 KB tiles: a K stage returns
// as soon as its score MMA has run, a V stage only after the chunk's P.V. Measured
// on batched Whisper-Base, two K and four V stages are fastest up to twelve query
// columns and three and three at sixteen.
constexpr int kRingTiles = 6;
template <int kNQT>
__host__ __device__ constexpr int k_stages() { return kNQT >= 16 ? 3 : 2; }
constexpr int kRingBytes = kRingTiles * kTileBytes;
constexpr int kPBytes = 4096;                  // P of a chunk: 128 keys x 16 queries x 2 B
constexpr int kQTileBytes = kSCols * kRowBytes; // 4 KB
constexpr int kConsumerWarps = 4;              // one key per consumer thread
constexpr int kThreads = (kConsumerWarps + 3) * 32;   // + producer, score-MMA and P.V-MMA warps
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMmaWarp = kConsumerWarps + 1;
constexpr int kPvWarp = kConsumerWarps + 2;
constexpr int kCtasPerSm = 2;
constexpr uint32_t kTmemCols = 128;            // S: 2 x 32 at 0; O^T: 2 x 16 (row segments) at 64
constexpr uint32_t kOCol = 64;
constexpr float kRescaleLog2 = 8.f;            // a reference max moves only past this margin (x256)
// K full/empty [K stages], V full/empty [V stages]; tfull, tempty, pempty, ofull, pfull [2]
constexpr int kRingBars = 2 * kRingTiles;
constexpr int kBars = kRingBars + 10;
constexpr int kPRegion = 2 * kPBytes;

struct TcParams {
  const float* Q;
  const int* key_len;
  float* out;
  float* part;
  unsigned int* counters;   // arrival counters (the four-column instance)
  unsigned int* status;
  int B, T, LH, LHc, lh0, nq, part_stride;
  float qscale;
};

// OR of a predicate over the threads of a named barrier, which it also is.
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
// 2^x on the SFU (ex2.approx, flush-to-zero): 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// The dense chunk numbering from key_len, by one warp: s_nch[b] chunks per row of
// slot b, s_first[b] the number of slot b's first chunk (s_first[B] = total) and,
// if s_kl is given, the key lengths clamped to [0, T]. Every CTA of both kernels
// computes the same numbering.
__device__ __forceinline__ void number_chunks(const int* key_len, int B, int T, int LH, int lane, long long* s_first,
                                              int* s_nch, int* s_kl) {
  long long run = 0;
  for (int base_b = 0; base_b < B; base_b += 32) {
    const int b = base_b + lane;
    int nch = 0;
    if (b < B) {
      const int kl = min(max(__ldg(key_len + b), 0), T);
      nch = (kl + kChunk - 1) / kChunk;
      s_nch[b] = nch;
      if (s_kl != nullptr) s_kl[b] = kl;
    }
    long long v = static_cast<long long>(nch) * LH;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (b < B) s_first[b] = run + v - static_cast<long long>(nch) * LH;
    run += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) s_first[B] = run;
}

// The smallest power of two >= n (n <= 32).
template <int n>
__host__ __device__ constexpr int pow2_at_least() {
  return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : n <= 8 ? 8 : n <= 16 ? 16 : 32;
}

// Warp sums of v[0..N) (padded with zeros to a power of two P), reduce-scattered:
// at each halving a lane keeps the half of its values that its lane bit selects and
// adds its partner's copy of that half, so P - 1 shuffles leave each lane one
// query's sum over the lanes differing in the top log2(P) bits (query *q), and
// 5 - log2(P) more add the rest. Lanes whose low 5 - log2(P) bits are zero hold the
// P distinct totals.
template <int N>
__device__ __forceinline__ float warp_sum_scatter(const float (&v)[N], int lane, int* q) {
  constexpr int P = pow2_at_least<N>();
  float cur[P];
#pragma unroll
  for (int j = 0; j < P; ++j) cur[j] = j < N ? v[j] : 0.f;
  int qi = 0;
#pragma unroll
  for (int n = P, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float keep = hi ? cur[j + n / 2] : cur[j];
      const float send = hi ? cur[j] : cur[j + n / 2];
      cur[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
    if (hi) qi += n / 2;
  }
#pragma unroll
  for (int off = 32 / P / 2; off >= 1; off >>= 1) cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], off);
  *q = qi;
  return cur[0];
}

// Cut rows merged in the kernel, at the end of each CTA's range (four query
// columns), or by the merge kernel (more).
template <int kNQT>
__host__ __device__ constexpr bool merge_in_kernel() { return kNQT <= 4; }

template <int kNQT>   // query columns the softmax handles (4, 8, 12 or 16 >= nq)
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_shared_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                            const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  constexpr int kKStages = k_stages<kNQT>();
  constexpr int kVStages = kRingTiles - kKStages;
  // layout: P^T x 2 | K tiles x kKStages | V tiles x kVStages | Q tile | small arrays
  const uint32_t p_base = base;
  const uint32_t k_base = base + kPRegion;
  const uint32_t v_base = k_base + kKStages * kTileBytes;
  const uint32_t q_base = base + kPRegion + kRingBytes;
  float* s_red = reinterpret_cast<float*>(bp + kPRegion + kRingBytes + kQTileBytes);  // [4][16]
  float* s_corr = s_red + kConsumerWarps * kNPad;                     // [16] factors of the last max update
  float* s_sum = s_corr + kNPad;                                      // [2][4][16] per-warp sums of a segment
  float* s_m = s_sum + 2 * kConsumerWarps * kNPad;                    // [2][16] references of a segment
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_m + 2 * kNPad);
  long long* s_first = reinterpret_cast<long long*>(bars + kBars);
  int* s_nch = reinterpret_cast<int*>(s_first + p.B + 1);
  int* s_kl = s_nch + p.B + (p.B & 1);                                 // key lengths, clamped to [0, T]
  volatile int* s_flags = reinterpret_cast<volatile int*>(s_kl + p.B + (p.B & 1));   // abort, last, tmem base
  auto kfull_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto kempty_bar = [&](int s) { return smem_u32(&bars[kKStages + s]); };
  auto vfull_bar = [&](int s) { return smem_u32(&bars[2 * kKStages + s]); };
  auto vempty_bar = [&](int s) { return smem_u32(&bars[2 * kKStages + kVStages + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[kRingBars + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[kRingBars + 2 + a]); };
  auto pempty_bar = [&](int a) { return smem_u32(&bars[kRingBars + 4 + a]); };
  auto ofull_bar = [&](int a) { return smem_u32(&bars[kRingBars + 6 + a]); };
  auto pfull_bar = [&](int a) { return smem_u32(&bars[kRingBars + 8 + a]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int LH = p.LH, nq = p.nq;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {   // chunk numbering from key_len (every CTA computes the same prefix)
    number_chunks(p.key_len, p.B, p.T, LH, lane, s_first, s_nch, s_kl);
    if (lane == 0) {
      s_flags[0] = 0;
      s_flags[1] = 0;
    }
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(kfull_bar(s), 1);
      mbar_init(kempty_bar(s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(vfull_bar(s), 1);
      mbar_init(vempty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kConsumerWarps);
      mbar_init(pempty_bar(a), 1);
      mbar_init(ofull_bar(a), 1);
      mbar_init(pfull_bar(a), 1);
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

  // Q, out and the workspace may belong to the previous grid; the cache and key_len
  // are read before it has finished (no decode writes them), so the producer warp
  // starts streaming without waiting.
  if (warp != kProducerWarp) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp < kConsumerWarps) {   // rows of slots without any valid key: out = 0
    const long long per_slot = static_cast<long long>(nq) * LH * (kDh / 4);
    for (long long i = static_cast<long long>(blockIdx.x) * (kConsumerWarps * 32) + threadIdx.x; i < p.B * per_slot;
         i += static_cast<long long>(gridDim.x) * (kConsumerWarps * 32))
      if (s_nch[static_cast<int>(i / per_slot)] == 0)
        reinterpret_cast<float4*>(p.out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  if (active && warp == kProducerWarp) {
    // ------------------------------------------------------------ producers
    // lane 0 streams the K tiles, lane 1 the V tiles: a K stage comes back as soon
    // as its score MMA has run, a V stage only after the chunk's P.V.
    if (lane < 2) {
      const bool v_ring = lane == 1;
      const void* tm = v_ring ? static_cast<const void*>(&tmV) : static_cast<const void*>(&tmK);
      Cursor cur = locate(g0, s_first, s_nch, p.B);
      uint32_t armed = 0, armed_parity = 0;
      bool ok = true;
      const int nst = v_ring ? kVStages : kKStages;
      for (long long g = g0, i = 0; g < g1; ++g, ++i) {
        const int s = static_cast<int>(i % nst);
        const uint32_t parity = static_cast<uint32_t>((i / nst) & 1);
        if (!mbar_wait(v_ring ? vempty_bar(s) : kempty_bar(s), parity ^ 1u, s_flags)) {
          ok = false;
          break;
        }
        const int kl = s_kl[cur.b];
        const int t0 = cur.c * kChunk;
        const int nbox = (min(kChunk, kl - t0) + kBoxRows - 1) / kBoxRows;   // rows past them stay stale
        const int crow = cur.b * p.LHc + p.lh0 + cur.lh;
        const uint32_t fb = v_ring ? vfull_bar(s) : kfull_bar(s);
        const uint32_t dst = (v_ring ? v_base : k_base) + s * kTileBytes;
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nbox * kBoxBytes));
        for (int j = 0; j < nbox; ++j) tma_load_3d(dst + j * kBoxBytes, tm, fb, 0, t0 + j * kBoxRows, crow);
        armed |= 1u << s;
        armed_parity = (armed_parity & ~(1u << s)) | (parity << s);
        advance(cur, s_nch, p.B, LH);
      }
      if (!ok) {
        s_flags[0] = 1;
        atomicOr(p.status, 1u);
        for (int s = 0; s < nst; ++s)
          if (armed & (1u << s)) mbar_wait(v_ring ? vfull_bar(s) : kfull_bar(s), (armed_parity >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (active && warp == kMmaWarp) {
    // ------------------------------------------------------------ Q tiles + score MMAs
    constexpr uint32_t idesc_s = make_idesc(1u, kChunk, kSCols);
    Cursor cur = locate(g0, s_first, s_nch, p.B);
    int prev_b = -1, prev_lh = -1;
    bool ok = true;
    // lane: query row (lane / 2), half (lane & 1) of its channels. The rows of the
    // next segment are loaded into registers while the current one runs.
    const int qr = lane >> 1, half = lane & 1;
    const bool q_valid = qr < nq;
    float4 qn[8];
    auto load_q = [&](int b, int lh) {
      const float* src = p.Q + qrow(b, lh, q_valid ? qr : 0) * kDh + half * 32;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        qn[j] = q_valid ? __ldg(reinterpret_cast<const float4*>(src) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    // the segment after the row (b, lh), whose chunk 0 is g, if this CTA's range reaches it
    auto load_next_segment = [&](int b, int lh, long long g) {
      if (g + s_nch[b] >= g1) return;
      if (++lh == LH) {
        lh = 0;
        do {
          ++b;
        } while (b < p.B && s_nch[b] == 0);
      }
      load_q(b, lh);
    };
    load_q(cur.b, cur.lh);
    for (long long g = g0, i = 0; g < g1; ++g, ++i) {
      const int s = static_cast<int>(i % kKStages);
      const int a = static_cast<int>(i & 1);
      if (!mbar_wait(tempty_bar(a), static_cast<uint32_t>(((i >> 1) & 1) ^ 1), s_flags)) {
        ok = false;
        break;
      }
      if (cur.b != prev_b || cur.lh != prev_lh) {
        // A new row segment: its queries become the B operand of the scores, as bf16
        // hi (rows 0..15) and lo (rows 16..31) parts: K.(hi + lo) carries Q to about
        // 16 mantissa bits. The single Q tile is rewritten once the previous chunk's
        // score MMA (and so every earlier one from this thread) has finished.
        if (i > 0 && !mbar_wait(tfull_bar(static_cast<int>((i - 1) & 1)), static_cast<uint32_t>(((i - 1) >> 1) & 1),
                                s_flags)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t wh[4], wl[4];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float4 f = qn[2 * j + k];
            const float x[4] = {f.x * p.qscale, f.y * p.qscale, f.z * p.qscale, f.w * p.qscale};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              __nv_bfloat162 hi = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
              __nv_bfloat162 lo = __floats2bfloat162_rn(x[2 * e] - __low2float(hi), x[2 * e + 1] - __high2float(hi));
              wh[2 * k + e] = *reinterpret_cast<uint32_t*>(&hi);
              wl[2 * k + e] = *reinterpret_cast<uint32_t*>(&lo);
            }
          }
          // a row is 128 bytes = 8 chunks of 8 bf16; this lane writes chunks 4*half .. 4*half+3
          const uint32_t chunk = static_cast<uint32_t>(4 * half + j);
          const int rl = qr + kNPad;
          st_shared_v4(q_base + qr * 128 + ((chunk ^ (qr & 7)) << 4), wh[0], wh[1], wh[2], wh[3]);
          st_shared_v4(q_base + rl * 128 + ((chunk ^ (rl & 7)) << 4), wl[0], wl[1], wl[2], wl[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        prev_b = cur.b;
        prev_lh = cur.lh;
        load_next_segment(cur.b, cur.lh, g - cur.c);
      }
      if (!mbar_wait(kfull_bar(s), static_cast<uint32_t>((i / kKStages) & 1), s_flags)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint64_t kd = smem_desc_k_sw128(k_base + s * kTileBytes);
        const uint64_t qd = smem_desc_k_sw128(q_base);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * kSCols);
#pragma unroll
        for (int k = 0; k < 4; ++k)   // +32 bytes along K per MMA: +2 in the address field
          mma_bf16(d_tmem, kd + 2 * k, qd + 2 * k, idesc_s, k != 0 ? 1u : 0u);
        tc_commit(tfull_bar(a));
        tc_commit(kempty_bar(s));
      }
      __syncwarp();
      advance(cur, s_nch, p.B, LH);
    }
    if (!ok) {
      s_flags[0] = 1;
      atomicOr(p.status, 1u);
    }
  } else if (active && warp == kPvWarp) {
    // ------------------------------------------------------------ P.V MMAs
    // Each chunk's P.V once its P^T and V tile are ready: A = the V tile (as V^T),
    // B = P^T, D = the row segment's O^T buffer (accumulating from its first chunk).
    if (lane == 0) {
      // A (V^T) and B (P^T, stored as P [key][query]) both MN-major
      constexpr uint32_t idesc_o = make_idesc(1u, kDh, kNPad) | (1u << 15) | (1u << 16);
      Cursor cur = locate(g0, s_first, s_nch, p.B);
      int prev_b = -1, prev_lh = -1, seg = -1;
      bool ok = true;
      for (long long g = g0, i = 0; g < g1; ++g, ++i) {
        const int b = static_cast<int>(i & 1), st = static_cast<int>(i % kVStages);
        const bool first = cur.b != prev_b || cur.lh != prev_lh;
        if (first) {
          ++seg;
          prev_b = cur.b;
          prev_lh = cur.lh;
        }
        const bool last = (cur.c == s_nch[cur.b] - 1) || (g + 1 == g1);
        if (!mbar_wait(pfull_bar(b), static_cast<uint32_t>((i >> 1) & 1), s_flags) ||
            !mbar_wait(vfull_bar(st), static_cast<uint32_t>((i / kVStages) & 1), s_flags)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int rb = seg & 1;
        const uint64_t vd = smem_desc_mn_sw128(v_base + st * kTileBytes);
        const uint64_t pd = smem_desc_mn_sw32(p_base + b * kPBytes);
        const uint32_t d_tmem = tmem_base + kOCol + static_cast<uint32_t>(rb * kNPad);
#pragma unroll
        for (int kb = 0; kb < kChunk / 16; ++kb)   // 16 keys: 2048 bytes of V, 512 bytes of P
          mma_bf16(d_tmem, vd + kb * (2048 >> 4), pd + kb * (512 >> 4), idesc_o, (first && kb == 0) ? 0u : 1u);
        tc_commit(pempty_bar(b));
        tc_commit(vempty_bar(st));
        if (last) tc_commit(ofull_bar(rb));
        advance(cur, s_nch, p.B, LH);
      }
      if (!ok) {
        s_flags[0] = 1;
        atomicOr(p.status, 1u);
      }
    }
    __syncwarp();
  } else if (active) {
    // ------------------------------------------------------------ consumers
    const int tid = threadIdx.x;                   // 0..127: key of the chunk for the softmax
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // this key's row of P [key][16 queries] (32 bytes) in buffer 0, and its swizzle:
    // queries 8j .. 8j + 7 go to 16-byte chunk j ^ ((tid >> 2) & 1)
    const uint32_t p_row = p_base + static_cast<uint32_t>(tid) * 32u;
    const uint32_t p_sw = static_cast<uint32_t>((tid >> 2) & 1);
    Cursor cur = locate(g0, s_first, s_nch, p.B);
    int seg_c0 = cur.c;
    // m_ref: the reference max the probabilities are taken against (log2 units); it
    // moves only when a score exceeds it by more than kRescaleLog2.
    float m_ref[kNQT], s_run[kNQT];
#pragma unroll
    for (int q = 0; q < kNQT; ++q) {
      m_ref[q] = -INFINITY;
      s_run[q] = 0.f;
    }
    bool ok = true;
    int seg = 0;          // index of the current row segment
    // A finished segment waiting to be written out (one chunk later, so that its
    // last P.V has run by then).
    bool f_pending = false, f_whole = false;
    int f_seg = 0, f_b = 0, f_lh = 0, f_pseg = 0, f_nseg = 1;
    // cut rows of this range, published at its end (in-kernel merge): slot, row, segments
    int n_cut = 0, cb0 = 0, clh0 = 0, cn0 = 0, cb1 = 0, clh1 = 0, cn1 = 0;
    long long f_row = 0;
    auto fail = [&]() {
      ok = false;
      s_flags[0] = 1;
      atomicOr(p.status, 1u);
    };
    // Write the finished segment f_seg: O^T from TMEM through a free P^T buffer
    // (as [query][channel] floats) to the output rows, or, for a part of a cut
    // row, to the segment's partial slots.
    auto flush = [&](int free_pbuf) {
      const int rb = f_seg & 1;
      if (ok && !mbar_wait(ofull_bar(rb), static_cast<uint32_t>((f_seg >> 1) & 1), s_flags)) fail();
      tc_fence_after();
      uint32_t o[16];
      tmem_ld_32x32b_x16(tmem_base + lane_base + kOCol + static_cast<uint32_t>(rb * kNPad), o);
      tmem_ld_wait();
      tc_fence_before();
      float* sO = reinterpret_cast<float*>(bp + free_pbuf * kPBytes);   // [16][64]
      if (lane < 16) {   // lane l of warp w: channel 16w + l
#pragma unroll
        for (int q = 0; q < kNQT; ++q) sO[q * kDh + 16 * warp + lane] = __uint_as_float(o[q]);
      }
      named_barrier(1, kConsumerWarps * 32);
      const float* sum = s_sum + rb * kConsumerWarps * kNPad;
      for (int e = tid; e < nq * (kDh / 4); e += kConsumerWarps * 32) {
        const int q = e / (kDh / 4), c4 = e % (kDh / 4);
        float4 v = *reinterpret_cast<const float4*>(sO + q * kDh + 4 * c4);
        if (f_whole) {
          const float S = sum[q] + sum[kNPad + q] + sum[2 * kNPad + q] + sum[3 * kNPad + q];
          const float inv = S > 0.f ? 1.f / S : 0.f;
          v = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
          if (ok) *reinterpret_cast<float4*>(p.out + qrow(f_b, f_lh, q) * kDh + 4 * c4) = v;
        } else {
          *reinterpret_cast<float4*>(p.part + ((f_row * nq + q) * p.part_stride + f_pseg) * kPartFloats + 4 +
                                     4 * c4) = ok ? v : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (!f_whole && tid < nq) {
        float* P = p.part + ((f_row * nq + tid) * p.part_stride + f_pseg) * kPartFloats;
        P[0] = ok ? s_m[rb * kNPad + tid] : -INFINITY;
        P[1] = ok ? sum[tid] + sum[kNPad + tid] + sum[2 * kNPad + tid] + sum[3 * kNPad + tid] : 0.f;
      }
      if (merge_in_kernel<kNQT>() && !f_whole) {   // only a range's first and last segments are cut
        if (n_cut == 0) {
          cb0 = f_b;
          clh0 = f_lh;
          cn0 = f_nseg;
        } else {
          cb1 = f_b;
          clh1 = f_lh;
          cn1 = f_nseg;
        }
        ++n_cut;
      }
      named_barrier(1, kConsumerWarps * 32);   // the staging buffer is free again
      f_pending = false;
    };

    // One pass past the range (tail) flushes the last segment, so that the flush,
    // the largest part of this code, is laid down once.
    long long i = 0;
    for (long long g = g0;; ++g, ++i) {
      const bool tail = g == g1;
      const int s = static_cast<int>(i % kVStages);
      const int a = static_cast<int>(i & 1);
      const uint32_t acc_parity = static_cast<uint32_t>((i >> 1) & 1);
      const int nch = tail ? 1 : s_nch[cur.b];
      const bool seg_ends = !tail && ((cur.c == nch - 1) || (g + 1 == g1));
      const int rb = seg & 1;
      if (!tail) {
      const int kl = s_kl[cur.b];
      const int n = min(kChunk, kl - cur.c * kChunk);
      const bool seg_first = cur.c == seg_c0;
      if (ok && !mbar_wait(tfull_bar(a), acc_parity, s_flags)) fail();
      tc_fence_after();
      uint32_t sh[16], sl[16];   // K.Q_hi, K.Q_lo
      tmem_ld_32x32b_x16(tmem_base + lane_base + static_cast<uint32_t>(a * kSCols), sh);
      tmem_ld_32x32b_x16(tmem_base + lane_base + static_cast<uint32_t>(a * kSCols + kNPad), sl);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(a));

      // ---- softmax of the chunk: thread tid owns key tid
      const bool valid_key = tid < n && ok;
      float sc[kNQT];
      bool need = false;
#pragma unroll
      for (int q = 0; q < kNQT; ++q) {
        sc[q] = valid_key ? __uint_as_float(sh[q]) + __uint_as_float(sl[q]) : -INFINITY;
        need |= sc[q] > m_ref[q] + kRescaleLog2;
      }
      bool rescale_o = false;
      if (named_barrier_or(1, kConsumerWarps * 32, need)) {
        // some score passed its reference by more than the margin: move every
        // reference to the running max (warp redux, then a 4-entry max)
        float mq[kNQT];
#pragma unroll
        for (int q = 0; q < kNQT; ++q) mq[q] = warp_max(sc[q]);
        if (lane == 0) {
#pragma unroll
          for (int q4 = 0; q4 < kNQT / 4; ++q4)
            *reinterpret_cast<float4*>(s_red + warp * kNPad + 4 * q4) =
                make_float4(mq[4 * q4], mq[4 * q4 + 1], mq[4 * q4 + 2], mq[4 * q4 + 3]);
        }
        named_barrier(1, kConsumerWarps * 32);
#pragma unroll
        for (int q = 0; q < kNQT; ++q) {
          float M = m_ref[q];
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, s_red[w * kNPad + q]);
          const float corr = m_ref[q] == -INFINITY ? 0.f : ex2(m_ref[q] - M);
          s_run[q] *= corr;
          if (tid == 0) s_corr[q] = corr;   // the same in every thread
          m_ref[q] = M;
        }
        rescale_o = !seg_first;
      }
      // the P^T buffer is free once the P.V of chunk i-2 has finished
      if (ok && !mbar_wait(pempty_bar(a), acc_parity ^ 1u, s_flags)) fail();
      {
        // the probabilities, rounded to bf16, eight queries to a 16-byte store
        uint32_t pw[(kNQT + 7) / 8 * 4];
#pragma unroll
        for (int q2 = 0; q2 < (kNQT + 7) / 8 * 4; ++q2) {
          float pr[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int q = 2 * q2 + e;
            pr[e] = q < kNQT && valid_key ? ex2(sc[q] - m_ref[q]) : 0.f;
          }
          // one conversion rounds both (queries 2 q2 in the low half, 2 q2 + 1 in the
          // high half); the sums add the rounded values, read back from the halves
          __nv_bfloat162 pp = __floats2bfloat162_rn(pr[0], pr[1]);
          const uint32_t u = *reinterpret_cast<uint32_t*>(&pp);
          if (2 * q2 < kNQT) s_run[2 * q2] += __uint_as_float(u << 16);
          if (2 * q2 + 1 < kNQT) s_run[2 * q2 + 1] += __uint_as_float(u & 0xFFFF0000u);
          pw[q2] = u;
        }
        const uint32_t row = p_row + static_cast<uint32_t>(a * kPBytes);
#pragma unroll
        for (int j = 0; j < (kNQT + 7) / 8; ++j)
          st_shared_v4(row + ((static_cast<uint32_t>(j) ^ p_sw) << 4), pw[4 * j], pw[4 * j + 1], pw[4 * j + 2],
                       pw[4 * j + 3]);
      }
      if (n < kChunk) {
        // tail chunk: zero the V rows of keys >= n (their P is 0; the rows may hold any bits)
        if (ok && !mbar_wait(vfull_bar(s), static_cast<uint32_t>((i / kVStages) & 1), s_flags)) fail();
        const uint32_t vt = v_base + s * kTileBytes;
        for (int u = n * (kRowBytes / 16) + tid; u < kTileBytes / 16; u += kConsumerWarps * 32)
          st_shared_v4(vt + u * 16, 0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      named_barrier(1, kConsumerWarps * 32);                 // P^T (and the V tail) complete
      if (rescale_o) {
        // O^T (chunks before this one) *= corr per query column, after their P.V and
        // before this chunk's; each warp scales its own 16 channel lanes
        if (ok && !mbar_wait(pempty_bar(a ^ 1), static_cast<uint32_t>(((i - 1) >> 1) & 1), s_flags)) fail();
        tc_fence_after();
        uint32_t o[16];
        tmem_ld_32x32b_x16(tmem_base + lane_base + kOCol + static_cast<uint32_t>(rb * kNPad), o);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < kNQT; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * s_corr[q]);
        tmem_st_32x32b_x16(tmem_base + lane_base + kOCol + static_cast<uint32_t>(rb * kNPad), o);
        tmem_st_wait();
        tc_fence_before();
        named_barrier(1, kConsumerWarps * 32);
      }
      if (tid == 0) mbar_arrive(pfull_bar(a));               // the MMA warp issues this chunk's P.V
      }
      // the previous segment's P.V has run by now; its P^T buffer (the other one) stages O.
      // Past the range every P.V has been issued, and both buffers are free once it has run.
      if (f_pending) flush(tail ? 0 : (a ^ 1));
      if (tail) break;

      if (seg_ends) {
        // ---- the segment ends: per-warp sums over the keys, references; written out next chunk
        if constexpr (kNQT < 16) {   // reduce-scattered (measured faster up to twelve columns)
          int qs;
          const float tot = warp_sum_scatter(s_run, lane, &qs);
          constexpr int kLanesPerQ = 32 / pow2_at_least<kNQT>();
          if ((lane & (kLanesPerQ - 1)) == 0 && qs < kNQT) s_sum[(rb * kConsumerWarps + warp) * kNPad + qs] = tot;
        } else {                     // a butterfly per query (faster at sixteen)
#pragma unroll
          for (int q = 0; q < kNQT; ++q) {
            float sq = s_run[q];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
            s_run[q] = sq;
          }
          if (lane == 0) {
#pragma unroll
            for (int q4 = 0; q4 < kNQT / 4; ++q4)
              *reinterpret_cast<float4*>(s_sum + (rb * kConsumerWarps + warp) * kNPad + 4 * q4) =
                  make_float4(s_run[4 * q4], s_run[4 * q4 + 1], s_run[4 * q4 + 2], s_run[4 * q4 + 3]);
          }
        }
        if (tid == 0) {   // the references are the same in every thread
#pragma unroll
          for (int q = 0; q < kNQT; ++q) s_m[rb * kNPad + q] = m_ref[q];
        }
        f_pending = true;
        f_seg = seg;
        f_b = cur.b;
        f_lh = cur.lh;
        f_row = static_cast<long long>(cur.b) * LH + cur.lh;
        f_whole = seg_c0 == 0 && cur.c == nch - 1;
        f_pseg = 0;
        f_nseg = 1;
        if (!f_whole) {   // this CTA's segment index among the row's owners, and their number
          const long long grow = s_first[cur.b] + static_cast<long long>(cur.lh) * nch;
          const long long first_owner = owner_of(grow, total, ranges);
          f_pseg = static_cast<int>(blockIdx.x - first_owner);
          f_nseg = static_cast<int>(owner_of(grow + nch - 1, total, ranges) - first_owner + 1);
        }
        ++seg;
#pragma unroll
        for (int q = 0; q < kNQT; ++q) {
          m_ref[q] = -INFINITY;
          s_run[q] = 0.f;
        }
      }
      const int pb = cur.b, plh = cur.lh;
      advance(cur, s_nch, p.B, LH);
      if (cur.b != pb || cur.lh != plh) seg_c0 = cur.c;
    }
    if (merge_in_kernel<kNQT>() && n_cut > 0) {
      // Publish the cut rows (their partial writes are ordered before this point by
      // the flushes' barriers) with acquire-release arrival counters; the last
      // arriver of a row merges its segments' states in segment order, after the
      // barrier that orders thread 0's acquire before every thread's reads.
      if (tid == 0) {
        const unsigned int prev0 = atomic_add_acq_rel_gpu(p.counters + static_cast<long long>(cb0) * LH + clh0, 1u);
        const unsigned int prev1 =
            n_cut > 1 ? atomic_add_acq_rel_gpu(p.counters + static_cast<long long>(cb1) * LH + clh1, 1u) : 0u;
        int last = prev0 == static_cast<unsigned int>(cn0 - 1) ? 1 : 0;
        if (n_cut > 1 && prev1 == static_cast<unsigned int>(cn1 - 1)) last |= 2;
        s_flags[1] = last;
      }
      named_barrier(1, kConsumerWarps * 32);
      const int last = s_flags[1];
      for (int k = 0; k < 2; ++k) {
        if (!(last & (1 << k))) continue;
        const int mb = k ? cb1 : cb0, mlh = k ? clh1 : clh0, nseg = k ? cn1 : cn0;
        const long long row = static_cast<long long>(mb) * LH + mlh;
#pragma unroll 2
        for (int e = tid; e < nq * kDh; e += kConsumerWarps * 32) {   // (query, channel)
          const int q = e / kDh, c = e % kDh;
          const float* P0 = p.part + (row * nq + q) * p.part_stride * kPartFloats;
          float MM = -INFINITY, SS = 0.f, AA = 0.f;
          for (int k0 = 0; k0 < nseg; k0 += 4) {
            float mk[4], sk[4], ak[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const bool in = k0 + u < nseg;
              const float* Pk = P0 + (k0 + u) * kPartFloats;
              mk[u] = in ? __ldcg(Pk) : -INFINITY;
              sk[u] = in ? __ldcg(Pk + 1) : 0.f;
              ak[u] = in ? __ldcg(Pk + 4 + c) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float M2 = fmaxf(MM, mk[u]);
              const float f0 = rescale(MM, M2), f1 = rescale(mk[u], M2);
              SS = SS * f0 + sk[u] * f1;
              AA = AA * f0 + ak[u] * f1;
              MM = M2;
            }
          }
          p.out[qrow(mb, mlh, q) * kDh + c] = SS > 0.f ? AA / SS : 0.f;
        }
        if (tid == 0) p.counters[row] = 0u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Rows cut by the boundaries of the main grid's ranges: the segment states that the
// CTAs sharing such a row left in its partial slots ((max, sum) and the unnormalised
// accumulator per query), merged in segment order into the output rows. One CTA per
// boundary; a row cut by several boundaries is merged at its first. Thread layout:
// the queries (padded to a power of two) split the CTA's threads; each thread takes
// one query and 1, 2 or 4 adjacent channels (one vector load per segment), so a
// segment's weight is one exp2 per query and thread, and its accumulator one fma
// per channel.
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads) decode_shared_merge_kernel(const TcParams p, int main_grid) {
  extern __shared__ uint8_t merge_smem[];
  long long* s_first = reinterpret_cast<long long*>(merge_smem);   // [B + 1]
  int* s_nch = reinterpret_cast<int*>(s_first + p.B + 1);           // [B]
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int LH = p.LH, nq = p.nq;
  if (threadIdx.x < 32) number_chunks(p.key_len, p.B, p.T, LH, lane, s_first, s_nch, nullptr);
  // Every CTA waits for the main grid, whether or not it has a row to merge: the
  // next grid's dependency wait, which covers this grid, then covers that one too.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  const long long total = s_first[p.B];
  const long long ranges = total < main_grid ? total : static_cast<long long>(main_grid);
  const int nqp = nq <= 1 ? 1 : nq <= 2 ? 2 : nq <= 4 ? 4 : nq <= 8 ? 8 : 16;
  const int tq = kMergeThreads / nqp;                 // threads per query
  const int q = threadIdx.x / tq, t = threadIdx.x % tq;
  const int cpt = tq >= kDh ? 1 : kDh / tq;           // channels t * cpt .. + cpt (<= 4)
  for (long long j = 1 + blockIdx.x; j < ranges; j += gridDim.x) {
    const long long g = j * total / ranges;   // first chunk of range j
    const Cursor cur = locate(g, s_first, s_nch, p.B);
    if (cur.c == 0) continue;                 // the boundary falls between rows
    const long long grow = g - cur.c;         // the row's first chunk
    if ((j - 1) * total / ranges > grow) continue;   // cut before, inside the row too
    if (q >= nq || t >= kDh) continue;
    const int nch = s_nch[cur.b];
    const long long first_owner = owner_of(grow, total, ranges);
    const int nseg = static_cast<int>(owner_of(grow + nch - 1, total, ranges) - first_owner + 1);
    const long long row = static_cast<long long>(cur.b) * LH + cur.lh;
    const float* P0 = p.part + (row * nq + q) * p.part_stride * kPartFloats;
    float MM = -INFINITY, SS = 0.f, AA[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < nseg; k0 += 4) {   // four segments' loads in flight at a time
      float mk[4], sk[4], ak[4][4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const bool in = k0 + v < nseg;
        const float* Pk = P0 + (k0 + v) * kPartFloats;
        mk[v] = in ? __ldcg(Pk) : -INFINITY;
        sk[v] = in ? __ldcg(Pk + 1) : 0.f;
        const float* a = Pk + 4 + t * cpt;   // 16-byte aligned for 4 channels, 8 for 2
        float4 av = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in) {
          if (cpt == 4) {
            av = __ldcg(reinterpret_cast<const float4*>(a));
          } else if (cpt == 2) {
            const float2 a2 = __ldcg(reinterpret_cast<const float2*>(a));
            av.x = a2.x;
            av.y = a2.y;
          } else {
            av.x = __ldcg(a);
          }
        }
        ak[v][0] = av.x;
        ak[v][1] = av.y;
        ak[v][2] = av.z;
        ak[v][3] = av.w;
      }
      float M = MM;
#pragma unroll
      for (int v = 0; v < 4; ++v) M = fmaxf(M, mk[v]);
      const float f0 = MM == -INFINITY ? 0.f : ex2(MM - M);
      float w[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) w[v] = mk[v] == -INFINITY ? 0.f : ex2(mk[v] - M);
      SS *= f0;
#pragma unroll
      for (int v = 0; v < 4; ++v) SS = fmaf(sk[v], w[v], SS);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        AA[c] *= f0;
#pragma unroll
        for (int v = 0; v < 4; ++v) AA[c] = fmaf(ak[v][c], w[v], AA[c]);
      }
      MM = M;
    }
    const float inv = SS > 0.f ? 1.f / SS : 0.f;
    float* o = p.out + ((static_cast<long long>(cur.b) * nq + q) * LH + cur.lh) * kDh + t * cpt;
    if (cpt == 4)
      *reinterpret_cast<float4*>(o) = make_float4(AA[0] * inv, AA[1] * inv, AA[2] * inv, AA[3] * inv);
    else if (cpt == 2)
      *reinterpret_cast<float2*>(o) = make_float2(AA[0] * inv, AA[1] * inv);
    else
      o[0] = AA[0] * inv;
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
  size_t n = 1024 + kPRegion + kRingBytes + kQTileBytes;
  n += (kConsumerWarps * kNPad + kNPad + 2 * kConsumerWarps * kNPad + 2 * kNPad) * 4 + kBars * 8;
  n += static_cast<size_t>(B + 1) * 8 + 2 * static_cast<size_t>(B + (B & 1)) * 4 + 16;
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
                      cudaStream_t stream, std::string* msg, int* grid) {
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
  cudaError_t e = cudaSuccess;
  {   // the occupancy of the last shared-memory size queried, per device
    static size_t occ_bytes[128] = {};
    static int occ_ctas[128] = {};
    std::lock_guard<std::mutex> lock(mu);
    const int d = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
    if (occ_bytes[d] != smem) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_shared_tc_kernel<kNQT>, kThreads, smem);
      if (e != cudaSuccess) return e;
      occ_bytes[d] = smem;
      occ_ctas[d] = per_sm;
    }
    per_sm = occ_ctas[d];
  }
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  if (per_sm < kCtasPerSm) {
    // The occupancy query reports one CTA per SM for kernels that allocate tensor
    // memory. Two of these fit by registers, shared memory and TMEM columns
    // (2 x 128 of 512), and no CTA waits on another, so the count is taken from
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
  *grid = dev.num_sms * (per_sm < kCtasPerSm ? per_sm : kCtasPerSm);
  cfg.gridDim = dim3(*grid);
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

// The merge kernel after a main grid of main_grid CTAs: one CTA per range boundary
// (main_grid - 1 of them at most), started by programmatic dependent launch so that
// its chunk numbering overlaps the main grid's tail.
cudaError_t launch_merge(const TcParams& prm, int main_grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(main_grid > 1 ? main_grid - 1 : 1);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(prm.B + 1) * 8 + static_cast<size_t>(prm.B) * 4;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_shared_merge_kernel, prm, main_grid);
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
  // the workspace has the stream kernel's layout: arrival counters (used by the
  // four-column instance, which leaves them at zero), then the partial slots
  int grid = 0;
  cudaError_t e = a.nq <= 4   ? launch_tc<4>(prm, a.Kc, a.Vc, dev, stream, msg, &grid)
                  : a.nq <= 8 ? launch_tc<8>(prm, a.Kc, a.Vc, dev, stream, msg, &grid)
                  : a.nq <= 12 ? launch_tc<12>(prm, a.Kc, a.Vc, dev, stream, msg, &grid)
                              : launch_tc<16>(prm, a.Kc, a.Vc, dev, stream, msg, &grid);
  if (e != cudaSuccess) return e;
  count_launches(1);
  if (!merge_in_kernel<4>() || a.nq > 4) {
    e = launch_merge(prm, grid, stream);
    if (e == cudaSuccess) count_launches(1);
  }
  return e;
}

}  // namespace cxa
