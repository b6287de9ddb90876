// Decode: query rows attend non-causally over the valid encoder keys of the
// projection cache, out = softmax(scale * q.K^T) V ("Whisper: Trace One Encoder
// Tensor into Every Decoder Layer", "View 2 -- expand one cross-attention
// operation": one query token, all key tokens, head_dim 64, scale 0.125).
// cxa_decode has one query row per (slot, layer, head); cxa_decode_shared has nq
// query rows (beam or speculative hypotheses) per (slot, layer, head) that all
// attend the same cache slot, the batch-N-queries-over-one-shared-cache case of
// SharedSplitKVCached ("Caso de estudio: WhisperKit", §3): each K/V row is read
// from HBM once and used for all nq queries.
//
// Split-T decoding with the lazy (online) softmax of SplitKV (same page, §3),
// laid out for an HBM-bound GPU:
//
//  * Work = every valid key of every cache row, cut into chunks of kChunkKeys
//    keys (16 KB of K and 16 KB of V). The chunks of all rows are numbered
//    densely, slot-major then (layer, head) then key order, and the persistent
//    grid gives each CTA one contiguous, equal-sized range of chunk numbers, so
//    every CTA streams the same number of bytes whatever the key lengths are.
//  * In each CTA a producer warp keeps a kStages-deep ring of shared-memory
//    stages full with cp.async.bulk copies per chunk (K rows, V rows and the
//    row's query rows, all contiguous) completing on a "full" mbarrier; the
//    consumer warps read a stage and release it on its "empty" mbarrier. The
//    copies of a stage are issued from separate lanes (one thread's bulk copies
//    are processed one after another).
//  * Each consumer lane group (16 lanes per fp32 key row, 8 or 16 per bf16 row)
//    runs its own online softmax per query (running max m, sum s, accumulators)
//    over the keys it is given, in fp32 and base 2 (q is pre-multiplied by
//    scale * log2(e)). With an fp32 cache and four or more queries a warp
//    instead takes 32 keys and half of the queries: register-tiled scores (a
//    4-key x query x 16-channel tile per lane, reduced to one key per lane),
//    the probabilities through shared memory, four channels per lane for P.V.
//  * When a row's run of chunks in this CTA ends, the groups' states are merged
//    (warp shuffles, then shared memory). A CTA that owned the whole row writes
//    out directly; otherwise it stores its partials (m, s, acc[64]), one per
//    query, and counts itself on the row's arrival counter, and the CTA that
//    arrives last merges the row's partials (M = max m_i, S = sum s_i 2^(m_i - M),
//    out = sum acc_i 2^(m_i - M) / S) and resets the counter. No CTA ever waits
//    for another CTA.
//  * Keys t >= key_len[b] are never copied and never enter the arithmetic; a
//    row with no valid key gets out = 0 (the clamped softmax denominator,
//    WhisperKit case study §2).
//  * Programmatic dependent launch: the next decode grid on the stream starts
//    streaming K/V while this one drains; it waits for this grid before
//    reading queries or writing anything.
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
constexpr int kPartFloats = 68;        // m, s, 2 pad, acc[64]
constexpr int kPartChunk = 64;         // partial-slot granularity of the workspace layout
// Launch shape (compile-time; the defaults were chosen by timing on GB300).
#ifndef CXA_DECODE_CONSUMER_WARPS
#define CXA_DECODE_CONSUMER_WARPS 4
#endif
#ifndef CXA_DECODE_STAGES          // ring depth of the 2-stage shape (more queries, self-attention, long streams)
#define CXA_DECODE_STAGES 2
#endif
#ifndef CXA_DECODE_STAGES_1Q       // ring depth with one or two queries per cache row
#define CXA_DECODE_STAGES_1Q 3
#endif
#ifndef CXA_DECODE_CHUNK_F32
#define CXA_DECODE_CHUNK_F32 64
#endif
#ifndef CXA_DECODE_CHUNK_BF16
#define CXA_DECODE_CHUNK_BF16 128
#endif
#ifndef CXA_DECODE_CTAS_PER_SM     // CTAs per SM of the 2-stage shape
#define CXA_DECODE_CTAS_PER_SM 3
#endif
#ifndef CXA_DECODE_CTAS_PER_SM_1Q  // CTAs per SM with one or two queries
#define CXA_DECODE_CTAS_PER_SM_1Q 2
#endif
#ifndef CXA_DECODE_PDL
#define CXA_DECODE_PDL 1
#endif
constexpr int kConsumerWarps = CXA_DECODE_CONSUMER_WARPS;
constexpr int kProducerWarp = kConsumerWarps;       // streams K/V (and Q) into the ring
constexpr int kMergeWarp = kConsumerWarps + 1;      // finishes the rows (output or split-row merge)
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kQRowBytes = kDh * 4;
static_assert(kConsumerWarps >= 1, "at least one consumer warp");

template <bool kBF16, int kNQ, bool kAppend = false, bool kShallow = false>
struct Traits {
  static constexpr int kElemBytes = kBF16 ? 2 : 4;
  static constexpr int kRowBytes = kDh * kElemBytes;                 // 256 / 128
  // One query: 8 lanes per bf16 row (16-byte slices). Several queries (fp32): 16
  // lanes per row, halving the per-lane query and accumulator registers.
  static constexpr int kLanesPerRow = (kBF16 && kNQ == 1) ? 8 : 16;
  static constexpr int kSliceBytes = kRowBytes / kLanesPerRow;       // 16 or 8
  static constexpr int kRowsPerPass = 32 / kLanesPerRow;             // keys per warp pass
  static constexpr int kElemsPerLane = kSliceBytes / kElemBytes;     // channels per lane
  static constexpr int kChunkKeys = kBF16 ? CXA_DECODE_CHUNK_BF16 : CXA_DECODE_CHUNK_F32;   // 16 KB of K
  // one or two queries: a deeper ring in fewer CTAs, so the slowest CTA, which ends
  // the launch, is relatively nearer the mean; the self-attention step (short rows,
  // one step after another) and very long streams (kShallow) keep more CTAs
  static constexpr bool kDeep = kNQ <= 2 && !kAppend && !kShallow;
  static constexpr int kStages = kDeep ? CXA_DECODE_STAGES_1Q : CXA_DECODE_STAGES;
  // fp32 cache with four or more queries: scores with one key per lane (no shuffles)
  static constexpr bool kKeyLanes = !kBF16 && kNQ >= 4;
  static constexpr int kPFloats = kKeyLanes ? kConsumerWarps * 32 * (kNQ / 2) : 0;   // probabilities
  // per query, the states a row end leaves for the merge warp: one per consumer warp,
  // or one per key half when the warps split the queries
  static constexpr int kSlotWarps = kKeyLanes ? 2 : kConsumerWarps;
  static constexpr int kKVBytes = kChunkKeys * kRowBytes;
  static constexpr int kStageBytes = 2 * kKVBytes + kNQ * kQRowBytes;
  static constexpr int kKeysPerWarp = kChunkKeys / kConsumerWarps;
  static constexpr int kPasses = kKeysPerWarp / kRowsPerPass;
  // passes whose scores are held at once (bounds the score registers to 16)
  static constexpr int kPassBlock = kPasses < 16 / kNQ ? kPasses : 16 / kNQ;
  static_assert(kPasses >= 1 && kKeysPerWarp % kRowsPerPass == 0, "chunk must split evenly over warps");
  static_assert(kPasses % kPassBlock == 0, "pass blocks must tile the passes");
  static_assert(kChunkKeys >= kPartChunk, "a row then has at most ceil(T / 64) segments: one partial slot each");
};

struct DecodeParams {
  const float* Q;
  const uint8_t* Kc;
  const uint8_t* Vc;
  const int* key_len;
  float* out;
  float* part;
  unsigned int* counters;
  unsigned int* status;
  int B, T, LH;        // LH = rows per slot in this call (layers [l0, l0+nl) x H)
  int LHc;             // rows per slot in the cache (L x H)
  int lh0;             // first cache row of the call within a slot (l0 x H)
  int nq;              // query rows per cache row (<= kNQ)
  int key_len_add;     // valid keys = clamp(key_len[b] + key_len_add, 0, T)
  int part_stride;     // partial slots per (row, query) (ceil(T / 64))
  float qscale;        // scale * log2(e)
  const float* Knew;   // kAppend: [B][L][H][64] rows for position key_len[b] (fp32)
  const float* Vnew;
};

// kAppend: the new row of each (slot, layer, head) at its position, as the lane
// slice of a cache row holds it (rounded to the cache dtype).
template <bool kBF16, int kEPL>
__device__ __forceinline__ void load_new_slice(const float* src, float* f) {
#pragma unroll
  for (int e4 = 0; e4 < kEPL / 4; ++e4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(src) + e4);
    f[4 * e4 + 0] = v.x;
    f[4 * e4 + 1] = v.y;
    f[4 * e4 + 2] = v.z;
    f[4 * e4 + 3] = v.w;
  }
  if constexpr (kBF16) {
#pragma unroll
    for (int e = 0; e < kEPL; ++e) f[e] = __bfloat162float(__float2bfloat16_rn(f[e]));
  }
}

// One lane's 16-byte slice of a cache row -> fp32 values (8 bf16 or 4 fp32)
template <bool kBF16, int kSlice>
__device__ __forceinline__ void load_slice(const uint8_t* p, float* f) {
  static_assert(kSlice == 16, "16-byte slices");
  const uint4 u = *reinterpret_cast<const uint4*>(p);
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

// Maximum over the warp's 32 lanes.
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Programmatic dependent launch: let the next grid on the stream be scheduled
// as this grid's CTAs retire, and wait for the previous grid to complete (and
// its memory to be visible) before touching anything it may have written.
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <bool kBF16, int kNQ, bool kAppend, bool kShallow = false>
constexpr int min_ctas_per_sm() {
  if (kNQ <= 2 && !kAppend && !kShallow) return CXA_DECODE_CTAS_PER_SM_1Q;
  if (!kBF16 && kNQ == 4) return 3;   // key-lane consumers: registers and shared memory fit three
  return kNQ >= 4 ? 2 : CXA_DECODE_CTAS_PER_SM;
}

// kAppend (self-attention step): the kernel also writes each row's new K/V at
// position key_len[b] (when in [0, T)) and attends positions 0 .. key_len[b]; the
// lane that meets that key takes it from Knew/Vnew rather than the cache copy it
// streamed, so nothing in the grid waits for the writes. The previous step wrote
// row pos - 1, so only chunks of keys below min(pos, T) - 1 are streamed before the
// grid dependency wait, and this instance lets the next grid start only after its
// own wait.
template <bool kBF16, int kNQ, bool kAppend = false, bool kShallow = false>
__global__ void __launch_bounds__(kThreads, (min_ctas_per_sm<kBF16, kNQ, kAppend, kShallow>()))
    decode_stream_kernel(const DecodeParams p) {
  using R = Traits<kBF16, kNQ, kAppend, kShallow>;
  constexpr int LPR = R::kLanesPerRow;
  constexpr int EPL = R::kElemsPerLane;

  constexpr int kStages = R::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  // full[S], empty[S], then the two row-end slots' rfull[2] (consumers -> merge warp)
  // and rfree[2] (merge warp -> consumers)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * R::kStageBytes);
  uint64_t* rbars = bars + 2 * kStages;
  long long* s_first = reinterpret_cast<long long*>(rbars + 4);
  int* s_nch = reinterpret_cast<int*>(s_first + p.B + 1);
  // a row end's per-warp states, double-buffered: slot k holds [kNQ][warps][64] acc,
  // [kNQ][warps] m, [kNQ][warps] s and [warps] ok
  constexpr int kSlotWarps = R::kSlotWarps;
  constexpr int kSlotFloats = kNQ * kSlotWarps * (kDh + 2) + kConsumerWarps;
  float* s_slots = reinterpret_cast<float*>(s_nch + p.B + (p.B & 1));
  volatile int* s_flags = reinterpret_cast<volatile int*>(s_slots + 2 * kSlotFloats);   // [0] abort
  // key-lane consumers: each warp's probabilities [32 keys][kNQ / 2]
  float* s_p = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(s_flags + 4) + 15) & ~static_cast<uintptr_t>(15));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int LH = p.LH;
  const int nq = p.nq;
  if constexpr (!kAppend) allow_dependent_launch();

  // ---- chunk numbering (every CTA computes the same prefix from key_len)
  if (warp == 0) {
    long long run = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      int nch = 0;
      if (b < p.B) {
        const int kl = min(max(__ldg(p.key_len + b) + p.key_len_add, 0), p.T);
        nch = (kl + R::kChunkKeys - 1) / R::kChunkKeys;
        s_nch[b] = nch;
      }
      long long v = static_cast<long long>(nch) * LH;   // inclusive warp scan
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
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[kStages + s]), kConsumerWarps);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&rbars[k]), kConsumerWarps);   // rfull[k]
      mbar_init(smem_u32(&rbars[2 + k]), 1);            // rfree[k]
    }
    fence_mbar_init();
  }
  __syncthreads();

  const long long total = s_first[p.B];
  const long long ranges = total < gridDim.x ? total : static_cast<long long>(gridDim.x);
  const bool active = total > 0 && blockIdx.x < ranges;
  const long long g0 = active ? blockIdx.x * total / ranges : 0;
  const long long g1 = active ? (blockIdx.x + 1) * total / ranges : 0;

  // The order in which the CTA works through its range: when the range ends inside a
  // row, that trailing segment [gA, g1) first, then [g0, gA). Both rows the CTA shares
  // with its neighbours are then finished, and merged by their last arriver, early,
  // behind the rest of the work, and the CTA ends on a whole row (a plain output
  // write). Position i of the sequence is chunk seq_g(i); step() moves a cursor on.
  long long gA = g1;
  if (active && g1 - g0 > 1) {
    const Cursor last = locate(g1 - 1, s_first, s_nch, p.B);
    if (last.c != s_nch[last.b] - 1 && (g1 - 1) - last.c > g0) gA = (g1 - 1) - last.c;
  }
  const long long nA = g1 - gA, nAll = g1 - g0;
  auto seq_g = [&](long long i) { return i < nA ? gA + i : g0 + (i - nA); };
  auto step = [&](Cursor& c, long long i) {   // from position i to i + 1
    if (i + 1 == nA) c = locate(g0, s_first, s_nch, p.B);
    else advance(c, s_nch, p.B, LH);
  };
  // the segment at position i ends there: the row's last chunk, or the end of a part
  auto seg_ends = [&](const Cursor& c, long long i) {
    return c.c == s_nch[c.b] - 1 || i + 1 == nA || i + 1 == nAll;
  };

  // The cache and key_len are inputs no decode writes: the producer starts
  // streaming the first stages' K and V rows before the previous grid is done.
  // The self-attention step (kAppend) reads early only the chunks whose keys all
  // lie below min(pos, T) - 1: the row at pos - 1 is the one the previous step
  // wrote, and that step (like this one) lets its successor start only after its
  // own dependency wait, so everything written before it is complete.
  const uint64_t pol = policy_evict_first();
  Cursor pcur{0, 0, 0};
  long long npre = 0, nissued = 0;
  // Stages [i0, i1) (at most kStages) go out from lane pairs of the producer warp:
  // lane 2(i - i0) arms stage i and copies its K rows, lane 2(i - i0) + 1 its V rows
  // (one thread's bulk copies are processed one after another, so a ring fill from
  // one thread would take a copy's turn per row block). c is the cursor of position
  // i0. Called by the whole producer warp.
  auto issue_stages = [&](long long i0, long long i1, Cursor c) {
    const long long i = i0 + (lane >> 1);
    const bool act = i < i1;
    for (long long k = i0; k < i && k < i1; ++k) step(c, k);
    uint32_t full = 0, dst = 0, kv_bytes = 0;
    size_t off = 0;
    if (act) {
      const int kl = min(max(__ldg(p.key_len + c.b) + p.key_len_add, 0), p.T);
      const int n = min(R::kChunkKeys, kl - c.c * R::kChunkKeys);
      const long long crow = static_cast<long long>(c.b) * p.LHc + p.lh0 + c.lh;   // cache row
      off = (static_cast<size_t>(crow) * p.T + static_cast<size_t>(c.c) * R::kChunkKeys) * R::kRowBytes;
      kv_bytes = static_cast<uint32_t>(n) * R::kRowBytes;
      full = smem_u32(&bars[i]);
      dst = smem_u32(stages + i * R::kStageBytes);
      if ((lane & 1) == 0) mbar_arrive_expect_tx(full, 2 * kv_bytes + static_cast<uint32_t>(nq) * kQRowBytes);
    }
    __syncwarp();
    if (act) {
      if ((lane & 1) == 0)
        bulk_g2s_hint(dst, p.Kc + off, kv_bytes, full, pol);
      else
        bulk_g2s_hint(dst + R::kKVBytes, p.Vc + off, kv_bytes, full, pol);
    }
  };
  Cursor pc{0, 0, 0};                    // kAppend: the first stage held back until the wait
  if (active && warp == kProducerWarp) {
    pcur = locate(seq_g(0), s_first, s_nch, p.B);
    npre = nAll < kStages ? nAll : kStages;
    long long pre_n = npre;
    if constexpr (kAppend) {
      Cursor c = pcur;
      for (pre_n = 0; pre_n < npre; ++pre_n) {
        const int kl = min(max(__ldg(p.key_len + c.b) + p.key_len_add, 0), p.T);
        const int end = c.c * R::kChunkKeys + min(R::kChunkKeys, kl - c.c * R::kChunkKeys);
        if (end > min(__ldg(p.key_len + c.b), p.T) - 1) break;   // may hold the previous step's row
        step(c, pre_n);
      }
      pc = c;
    }
    issue_stages(0, pre_n, pcur);
    nissued = pre_n;
  }
  if constexpr (kAppend) {
    wait_prior_grid();
    allow_dependent_launch();
    if (active && warp == kProducerWarp) {
      issue_stages(nissued, npre, pc);
      nissued = npre;
    }
  }
  // Q, out and the workspace may belong to the previous grid: wait for it.
  wait_prior_grid();
  // rows of slots without any valid key: out = 0
  {
    const long long per_slot = static_cast<long long>(nq) * LH * (kDh / 4);
    for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < p.B * per_slot;
         i += static_cast<long long>(gridDim.x) * kThreads) {
      if (s_nch[static_cast<int>(i / per_slot)] == 0)
        reinterpret_cast<float4*>(p.out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if constexpr (kAppend) {
    // the new rows into the cache: 16 lanes x 4 values per (slot, layer, head)
    const long long rows = static_cast<long long>(p.B) * LH;
    for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < rows * 16;
         i += static_cast<long long>(gridDim.x) * kThreads) {
      const long long row = i / 16;
      const int l16 = static_cast<int>(i % 16);
      const int b = static_cast<int>(row / LH), lh = static_cast<int>(row % LH);
      const int t = __ldg(p.key_len + b);
      if (t < 0 || t >= p.T) continue;
      const long long crow = static_cast<long long>(b) * p.LHc + p.lh0 + lh;
      const size_t dst = (static_cast<size_t>(crow) * p.T + t) * kDh + l16 * 4;
      const float4 k = __ldg(reinterpret_cast<const float4*>(p.Knew + crow * kDh) + l16);
      const float4 v = __ldg(reinterpret_cast<const float4*>(p.Vnew + crow * kDh) + l16);
      if constexpr (kBF16) {
        __nv_bfloat162 k01 = __floats2bfloat162_rn(k.x, k.y), k23 = __floats2bfloat162_rn(k.z, k.w);
        __nv_bfloat162 v01 = __floats2bfloat162_rn(v.x, v.y), v23 = __floats2bfloat162_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(const_cast<uint8_t*>(p.Kc) + dst * 2) =
            make_uint2(*reinterpret_cast<uint32_t*>(&k01), *reinterpret_cast<uint32_t*>(&k23));
        *reinterpret_cast<uint2*>(const_cast<uint8_t*>(p.Vc) + dst * 2) =
            make_uint2(*reinterpret_cast<uint32_t*>(&v01), *reinterpret_cast<uint32_t*>(&v23));
      } else {
        *reinterpret_cast<float4*>(const_cast<uint8_t*>(p.Kc) + dst * 4) = k;
        *reinterpret_cast<float4*>(const_cast<uint8_t*>(p.Vc) + dst * 4) = v;
      }
    }
  }
  if (!active) return;

  // query row n of cache row (b, lh): Q[b][n][lh][:]
  auto qrow = [&](int b, int lh, int n) { return (static_cast<long long>(b) * nq + n) * LH + lh; };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // The whole warp: lane 0 arms each stage, lanes 0 and 1 copy its K and V rows and
    // lanes 2 .. nq + 1 its query rows, so a stage's copies go out in parallel.
    Cursor cur = pcur;
    for (long long i = 0; i < npre; ++i) {   // the queries of the pre-issued stages
      const uint32_t qdst = smem_u32(stages + i * R::kStageBytes) + 2 * R::kKVBytes;
      const int qn = lane - static_cast<int>(i) * nq;
      if (qn >= 0 && qn < nq)
        bulk_g2s(qdst + qn * kQRowBytes, p.Q + qrow(cur.b, cur.lh, qn) * kDh, kQRowBytes, smem_u32(&bars[i]));
      step(cur, i);
    }
    uint32_t armed = static_cast<uint32_t>((1u << npre) - 1u), armed_parity = 0;
    bool ok = true;
    for (long long i = npre; i < nAll; ++i) {
      const int s = static_cast<int>(i % kStages);
      const uint32_t parity = static_cast<uint32_t>((i / kStages) & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[kStages + s]), parity ^ 1u, s_flags))) {
        ok = false;
        break;
      }
      const int kl = min(max(__ldg(p.key_len + cur.b) + p.key_len_add, 0), p.T);
      const int t0 = cur.c * R::kChunkKeys;
      const int n = min(R::kChunkKeys, kl - t0);
      const long long crow = static_cast<long long>(cur.b) * p.LHc + p.lh0 + cur.lh;   // cache row
      const size_t off = (static_cast<size_t>(crow) * p.T + t0) * R::kRowBytes;
      const uint32_t kv_bytes = static_cast<uint32_t>(n) * R::kRowBytes;
      const uint32_t full = smem_u32(&bars[s]);
      const uint32_t dst = smem_u32(stages + s * R::kStageBytes);
      if (lane == 0) mbar_arrive_expect_tx(full, 2 * kv_bytes + static_cast<uint32_t>(nq) * kQRowBytes);
      __syncwarp();
      if (lane == 0)
        bulk_g2s_hint(dst, p.Kc + off, kv_bytes, full, pol);
      else if (lane == 1)
        bulk_g2s_hint(dst + R::kKVBytes, p.Vc + off, kv_bytes, full, pol);
      else if (lane - 2 < nq)
        bulk_g2s(dst + 2 * R::kKVBytes + (lane - 2) * kQRowBytes, p.Q + qrow(cur.b, cur.lh, lane - 2) * kDh, kQRowBytes,
                 full);
      armed |= 1u << s;
      armed_parity = (armed_parity & ~(1u << s)) | (parity << s);
      step(cur, i);
    }
    if (!ok && lane == 0) {
      s_flags[0] = 1;
      atomicOr(p.status, 1u);
      for (int s = 0; s < kStages; ++s)   // let issued copies land before exiting
        if (armed & (1u << s)) mbar_wait(smem_u32(&bars[s]), (armed_parity >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == kMergeWarp) {
    // ------------------------------------------------------------ merge warp
    // Walks the same chunk sequence as the consumers; at each row end it takes the
    // consumers' states from slot re & 1, frees the slot, and writes the row (whole
    // rows) or its partial, the last arriver of a split row merging all partials.
    // Lane l owns channels l and l + 32.
    Cursor cur = locate(seq_g(0), s_first, s_nch, p.B);
    int seg_c0 = cur.c;
    int re = 0;
    for (long long i = 0; i < nAll; ++i) {
      const int nch = s_nch[cur.b];
      if (seg_ends(cur, i)) {
        const int slot = re & 1;
        bool okr = mbar_wait(smem_u32(&rbars[slot]), static_cast<uint32_t>((re >> 1) & 1), s_flags);
        if (!okr) {
          s_flags[0] = 1;
          if (lane == 0) atomicOr(p.status, 1u);
        }
        const float* sl_red = s_slots + slot * kSlotFloats;
        const float* sl_m = sl_red + kNQ * kSlotWarps * kDh;
        const float* sl_s = sl_m + kNQ * kSlotWarps;
        const float* sl_ok = sl_s + kNQ * kSlotWarps;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) okr = okr && sl_ok[w] != 0.f;
        float Mq[kNQ], Sq[kNQ], Aq[kNQ][2];
#pragma unroll
        for (int q = 0; q < kNQ; ++q) {
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < kSlotWarps; ++w) M = fmaxf(M, sl_m[q * kSlotWarps + w]);
          float S = 0.f, A0 = 0.f, A1 = 0.f;
#pragma unroll
          for (int w = 0; w < kSlotWarps; ++w) {
            const float f = rescale(sl_m[q * kSlotWarps + w], M);
            S = fmaf(sl_s[q * kSlotWarps + w], f, S);
            A0 = fmaf(sl_red[(q * kSlotWarps + w) * kDh + lane], f, A0);
            A1 = fmaf(sl_red[(q * kSlotWarps + w) * kDh + lane + 32], f, A1);
          }
          Mq[q] = M;
          Sq[q] = S;
          Aq[q][0] = A0;
          Aq[q][1] = A1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&rbars[2 + slot]));   // the slot may be rewritten
        ++re;
        const long long row = static_cast<long long>(cur.b) * LH + cur.lh;
        const bool whole_row = seg_c0 == 0 && cur.c == nch - 1;
        if (whole_row) {
#pragma unroll
          for (int q = 0; q < kNQ; ++q)
            if (q < nq && okr) {
              float* o = p.out + qrow(cur.b, cur.lh, q) * kDh;
              o[lane] = Sq[q] > 0.f ? Aq[q][0] / Sq[q] : 0.f;
              o[lane + 32] = Sq[q] > 0.f ? Aq[q][1] / Sq[q] : 0.f;
            }
        } else {
          const long long grow = s_first[cur.b] + static_cast<long long>(cur.lh) * nch;   // chunk 0 of row
          const long long first_owner = owner_of(grow, total, ranges);
          const int nseg = static_cast<int>(owner_of(grow + nch - 1, total, ranges) - first_owner + 1);
          const int seg = static_cast<int>(blockIdx.x - first_owner);
#pragma unroll
          for (int q = 0; q < kNQ; ++q) {
            if (q >= nq) continue;
            float* P = p.part + ((row * nq + q) * p.part_stride + seg) * kPartFloats;
            P[4 + lane] = okr ? Aq[q][0] : 0.f;
            P[4 + lane + 32] = okr ? Aq[q][1] : 0.f;
            if (lane == 0) {
              P[0] = okr ? Mq[q] : -INFINITY;
              P[1] = okr ? Sq[q] : 0.f;
            }
          }
          __syncwarp();   // orders every lane's partial writes before lane 0's release
          unsigned int last = 0u;
          if (lane == 0) {
            const unsigned int prev = atomic_add_acq_rel_gpu(p.counters + row, 1u);
            last = prev == static_cast<unsigned int>(nseg - 1) ? 1u : 0u;
          }
          if (__shfl_sync(0xffffffffu, last, 0)) {
            __syncwarp();   // lane 0's acquire before every lane's reads of the partials
            // the segments' states in segment order, rescaling as the max grows; four
            // queries by four segments of loads in flight at a time, and per query and
            // four segments one max and five exponentials (the old max's factor and the
            // segments' weights)
            constexpr int kQB = kNQ >= 6 ? 4 : (kNQ >= 2 ? 2 : 1);
            for (int q0 = 0; q0 < nq; q0 += kQB) {
              float MM[kQB], SS[kQB], A0[kQB], A1[kQB];
#pragma unroll
              for (int u = 0; u < kQB; ++u) {
                MM[u] = -INFINITY;
                SS[u] = 0.f;
                A0[u] = 0.f;
                A1[u] = 0.f;
              }
              for (int k0 = 0; k0 < nseg; k0 += 4) {
                float mk[kQB][4], sk[kQB][4], a0k[kQB][4], a1k[kQB][4];
#pragma unroll
                for (int u = 0; u < kQB; ++u) {
                  const float* P0 = p.part + (row * nq + (q0 + u < nq ? q0 + u : 0)) * p.part_stride * kPartFloats;
#pragma unroll
                  for (int v = 0; v < 4; ++v) {
                    const bool in = q0 + u < nq && k0 + v < nseg;
                    const float* Pk = P0 + (k0 + v) * kPartFloats;
                    mk[u][v] = in ? __ldcg(Pk) : -INFINITY;
                    sk[u][v] = in ? __ldcg(Pk + 1) : 0.f;
                    a0k[u][v] = in ? __ldcg(Pk + 4 + lane) : 0.f;
                    a1k[u][v] = in ? __ldcg(Pk + 4 + lane + 32) : 0.f;
                  }
                }
#pragma unroll
                for (int u = 0; u < kQB; ++u) {
                  float M = MM[u];
#pragma unroll
                  for (int v = 0; v < 4; ++v) M = fmaxf(M, mk[u][v]);
                  const float f0 = rescale(MM[u], M);
                  SS[u] *= f0;
                  A0[u] *= f0;
                  A1[u] *= f0;
#pragma unroll
                  for (int v = 0; v < 4; ++v) {
                    const float w = rescale(mk[u][v], M);
                    SS[u] = fmaf(sk[u][v], w, SS[u]);
                    A0[u] = fmaf(a0k[u][v], w, A0[u]);
                    A1[u] = fmaf(a1k[u][v], w, A1[u]);
                  }
                  MM[u] = M;
                }
              }
#pragma unroll
              for (int u = 0; u < kQB; ++u) {
                if (q0 + u < nq) {
                  float* o = p.out + qrow(cur.b, cur.lh, q0 + u) * kDh;
                  const float inv = SS[u] > 0.f ? 1.f / SS[u] : 0.f;
                  o[lane] = A0[u] * inv;
                  o[lane + 32] = A1[u] * inv;
                }
              }
            }
            if (lane == 0) p.counters[row] = 0u;
          }
        }
      }
      const int prev_b = cur.b, prev_lh = cur.lh;
      step(cur, i);
      if (cur.b != prev_b || cur.lh != prev_lh) seg_c0 = cur.c;
    }
  } else if constexpr (R::kKeyLanes) {
    // ------------------------------------------------------------ consumers, several
    // queries on an fp32 cache: warp w takes keys 32*(w & 1) .. +32 of each chunk and
    // queries (w >> 1)*QPW .. +QPW. Scores are register-tiled: lane (kq, cgh, cgl,
    // kg_lo) = lane bits (4, 3, 2, 1..0) accumulates a 4-key x QPW-query tile over the
    // 16 channels of channel group cg = 2 cgh + cgl, for the keys of key group
    // kg = 4 kq + kg_lo, each 16-byte slice read once for four keys or QPW queries.
    // The slices are visited in an order rotated by kg_lo, so the eight lanes of a
    // quarter warp (two channel groups x four rotations) read eight distinct bank
    // groups. A reduce-scatter over lane bits 2 and 3 then leaves each lane the QPW
    // whole scores of one key, 4 kg + 2 cgl + cgh. The probabilities go to shared
    // memory by key. P.V: lane (kp, cq) = lane bits (4, 3..0) takes the keys of parity
    // kp and channels 4cq .. 4cq + 3 (one 16-byte V slice and one probability
    // broadcast per key for 4 x QPW products); the two parities meet at the row end.
    constexpr int QPW = kNQ / 2;
    static_assert(kConsumerWarps == 4 && R::kChunkKeys == 64 && (QPW == 2 || QPW == 3 || QPW % 4 == 0),
                  "two key halves x two query halves of a 64-key chunk");
    const int kh = warp & 1, qh = warp >> 1;
    const int kg_lo = lane & 3, cgl = (lane >> 2) & 1, cgh = (lane >> 3) & 1;
    const int kg = (lane >> 4) * 4 + kg_lo;            // key group: keys 4kg .. 4kg + 3 of the half
    const int cg = cgh * 2 + cgl;                      // channel group: channels 16cg .. 16cg + 15
    const int my_key = kg * 4 + 2 * cgl + cgh;         // the key whose scores this lane ends with
    float* s_pw = s_p + warp * 32 * QPW;   // this warp's probabilities, [32 keys][QPW]
    const int kpar = lane >> 4, cq = lane & 15;       // P.V: key parity, channel quad
    Cursor cur = locate(seq_g(0), s_first, s_nch, p.B);
    float m[QPW], lsum[QPW], acc[QPW][4];
#pragma unroll
    for (int qi = 0; qi < QPW; ++qi) {
      m[qi] = -INFINITY;
      lsum[qi] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[qi][c] = 0.f;
    }
    bool ok = true;
    int re = 0;                          // row ends handed to the merge warp so far
    for (long long i = 0; i < nAll; ++i) {
      const int s = static_cast<int>(i % kStages);
      const uint32_t parity = static_cast<uint32_t>((i / kStages) & 1);
      if (ok && !mbar_wait(smem_u32(&bars[s]), parity, s_flags)) {
        ok = false;
        s_flags[0] = 1;
        atomicOr(p.status, 1u);
      }
      if (ok) {
        const int kl = min(max(__ldg(p.key_len + cur.b) + p.key_len_add, 0), p.T);
        const int n = min(R::kChunkKeys, kl - cur.c * R::kChunkKeys);
        const uint8_t* sK = stages + s * R::kStageBytes;
        const float* kp = reinterpret_cast<const float*>(sK + (kh * 32 + kg * 4) * R::kRowBytes) + cg * 16;
        const float* qp = reinterpret_cast<const float*>(sK + 2 * R::kKVBytes) + qh * QPW * kDh + cg * 16;
        float part[4][QPW];
#pragma unroll
        for (int jk = 0; jk < 4; ++jk)
#pragma unroll
          for (int qi = 0; qi < QPW; ++qi) part[jk][qi] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c4 = ((j + kg_lo) & 3) * 4;
          float4 kv[4];
#pragma unroll
          for (int jk = 0; jk < 4; ++jk) kv[jk] = *reinterpret_cast<const float4*>(kp + jk * kDh + c4);
#pragma unroll
          for (int qi = 0; qi < QPW; ++qi) {
            const float4 qv = *reinterpret_cast<const float4*>(qp + qi * kDh + c4);
#pragma unroll
            for (int jk = 0; jk < 4; ++jk) {
              part[jk][qi] = fmaf(qv.x, kv[jk].x, part[jk][qi]);
              part[jk][qi] = fmaf(qv.y, kv[jk].y, part[jk][qi]);
              part[jk][qi] = fmaf(qv.z, kv[jk].z, part[jk][qi]);
              part[jk][qi] = fmaf(qv.w, kv[jk].w, part[jk][qi]);
            }
          }
        }
        // reduce-scatter over the channel groups: lane bit 2 (cgl) keeps keys 2 cgl,
        // 2 cgl + 1 of the tile, then lane bit 3 (cgh) keeps key 2 cgl + cgh
        float half[2][QPW];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int qi = 0; qi < QPW; ++qi) {
            const float send = cgl ? part[t][qi] : part[2 + t][qi];
            const float keep = cgl ? part[2 + t][qi] : part[t][qi];
            half[t][qi] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
          }
        float sc[QPW];
#pragma unroll
        for (int qi = 0; qi < QPW; ++qi) {
          const float send = cgh ? half[0][qi] : half[1][qi];
          const float keep = cgh ? half[1][qi] : half[0][qi];
          sc[qi] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        const bool valid = kh * 32 + my_key < n;
        float pw[QPW];
#pragma unroll
        for (int qi = 0; qi < QPW; ++qi) {
          const float sv = valid ? sc[qi] * p.qscale : -INFINITY;
          const float mnew = fmaxf(m[qi], warp_max_f32(sv));
          const float corr = rescale(m[qi], mnew);   // 0 while the state is empty
          m[qi] = mnew;
          pw[qi] = valid ? exp2f(sv - mnew) : 0.f;
          lsum[qi] = fmaf(lsum[qi], corr, pw[qi]);
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[qi][c] *= corr;
        }
        if constexpr (QPW % 4 == 0) {
#pragma unroll
          for (int q4 = 0; q4 < QPW / 4; ++q4)
            *reinterpret_cast<float4*>(s_pw + my_key * QPW + 4 * q4) =
                make_float4(pw[4 * q4], pw[4 * q4 + 1], pw[4 * q4 + 2], pw[4 * q4 + 3]);
        } else if constexpr (QPW == 2) {
          *reinterpret_cast<float2*>(s_pw + my_key * QPW) = make_float2(pw[0], pw[1]);
        } else {
#pragma unroll
          for (int qi = 0; qi < QPW; ++qi) s_pw[my_key * QPW + qi] = pw[qi];
        }
        __syncwarp();
        const int nk = min(32, n - kh * 32);   // valid keys of this warp's half
        const float* vp = reinterpret_cast<const float*>(sK + R::kKVBytes + kh * 32 * R::kRowBytes) + 4 * cq;
#pragma unroll 4
        for (int k = kpar; k < nk; k += 2) {
          const float4 v4 = *reinterpret_cast<const float4*>(vp + k * kDh);
          float pk[QPW];
          if constexpr (QPW % 4 == 0) {
#pragma unroll
            for (int q4 = 0; q4 < QPW / 4; ++q4) {
              const float4 t = *reinterpret_cast<const float4*>(s_pw + k * QPW + 4 * q4);
              pk[4 * q4] = t.x;
              pk[4 * q4 + 1] = t.y;
              pk[4 * q4 + 2] = t.z;
              pk[4 * q4 + 3] = t.w;
            }
          } else if constexpr (QPW == 2) {
            const float2 t = *reinterpret_cast<const float2*>(s_pw + k * QPW);
            pk[0] = t.x;
            pk[1] = t.y;
          } else {
#pragma unroll
            for (int qi = 0; qi < QPW; ++qi) pk[qi] = s_pw[k * QPW + qi];
          }
#pragma unroll
          for (int qi = 0; qi < QPW; ++qi) {
            acc[qi][0] = fmaf(pk[qi], v4.x, acc[qi][0]);
            acc[qi][1] = fmaf(pk[qi], v4.y, acc[qi][1]);
            acc[qi][2] = fmaf(pk[qi], v4.z, acc[qi][2]);
            acc[qi][3] = fmaf(pk[qi], v4.w, acc[qi][3]);
          }
        }
      }
      __syncwarp();                      // the probabilities are rewritten by the next chunk
      if (lane == 0) mbar_arrive(smem_u32(&bars[kStages + s]));

      if (seg_ends(cur, i)) {
        // ---- hand the row's state to the merge warp: this warp's queries, at its
        //      key half's place in the slot
        const int slot = re & 1;
        if (re >= 2 && !mbar_wait(smem_u32(&rbars[2 + slot]), static_cast<uint32_t>(((re >> 1) - 1) & 1), s_flags)) {
          ok = false;                                      // the merge warp has not read this slot
          s_flags[0] = 1;
          atomicOr(p.status, 1u);
        }
        float* sl_red = s_slots + slot * kSlotFloats;
        float* sl_m = sl_red + kNQ * kSlotWarps * kDh;
        float* sl_s = sl_m + kNQ * kSlotWarps;
        float* sl_ok = sl_s + kNQ * kSlotWarps;
#pragma unroll
        for (int qi = 0; qi < QPW; ++qi) {
          const int q = qh * QPW + qi;
          float S = lsum[qi];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
          float a4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) a4[c] = acc[qi][c] + __shfl_xor_sync(0xffffffffu, acc[qi][c], 16);
          if (kpar == 0) {   // the slots are 8-byte aligned: two 8-byte stores
            float* dst = sl_red + (q * kSlotWarps + kh) * kDh + 4 * cq;
            *reinterpret_cast<float2*>(dst) = make_float2(a4[0], a4[1]);
            *reinterpret_cast<float2*>(dst + 2) = make_float2(a4[2], a4[3]);
          }
          if (lane == 0) {
            sl_m[q * kSlotWarps + kh] = m[qi];
            sl_s[q * kSlotWarps + kh] = S;
          }
        }
        if (lane == 0) sl_ok[warp] = ok ? 1.f : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&rbars[slot]));   // release: the slot's writes come first
        ++re;
#pragma unroll
        for (int qi = 0; qi < QPW; ++qi) {
          m[qi] = -INFINITY;
          lsum[qi] = 0.f;
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[qi][c] = 0.f;
        }
      }
      step(cur, i);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int sub = lane % LPR;          // slice of a key row this lane reads
    const int grp = lane / LPR;          // lane group = independent softmax stream
    Cursor cur = locate(seq_g(0), s_first, s_nch, p.B);
    int seg_c0 = cur.c;                  // first chunk of the current row segment
    float m[kNQ], ssum[kNQ], acc[kNQ][EPL];
#pragma unroll
    for (int q = 0; q < kNQ; ++q) {
      m[q] = -INFINITY;
      ssum[q] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[q][e] = 0.f;
    }
    bool ok = true;
    int re = 0;                          // row ends handed to the merge warp so far

    for (long long i = 0; i < nAll; ++i) {
      const int s = static_cast<int>(i % kStages);
      const uint32_t parity = static_cast<uint32_t>((i / kStages) & 1);
      if (ok && !mbar_wait(smem_u32(&bars[s]), parity, s_flags)) {
        ok = false;
        s_flags[0] = 1;
        atomicOr(p.status, 1u);
      }
      const int kl = min(max(__ldg(p.key_len + cur.b) + p.key_len_add, 0), p.T);
      const int n = min(R::kChunkKeys, kl - cur.c * R::kChunkKeys);
      int subst = -1;   // kAppend: the chunk row that is the new key
      const float* knew_row = nullptr;
      const float* vnew_row = nullptr;
      if constexpr (kAppend) {
        const int t = __ldg(p.key_len + cur.b) - cur.c * R::kChunkKeys;
        if (__ldg(p.key_len + cur.b) < p.T && t >= 0 && t < n) {
          subst = t;
          const long long crow = static_cast<long long>(cur.b) * p.LHc + p.lh0 + cur.lh;
          knew_row = p.Knew + crow * kDh + sub * EPL;
          vnew_row = p.Vnew + crow * kDh + sub * EPL;
        }
      }
      if (ok) {
        const uint8_t* sK = stages + s * R::kStageBytes;
        const uint8_t* sV = sK + R::kKVBytes;
        const float* sQ = reinterpret_cast<const float*>(sK + 2 * R::kKVBytes);
        float qv[kNQ][EPL];
#pragma unroll
        for (int q = 0; q < kNQ; ++q) {
          if (q < nq) {
#pragma unroll
            for (int e4 = 0; e4 < EPL / 4; ++e4) {
              const float4 v = *reinterpret_cast<const float4*>(sQ + q * kDh + sub * EPL + 4 * e4);
              qv[q][4 * e4 + 0] = v.x * p.qscale;
              qv[q][4 * e4 + 1] = v.y * p.qscale;
              qv[q][4 * e4 + 2] = v.z * p.qscale;
              qv[q][4 * e4 + 3] = v.w * p.qscale;
            }
          } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) qv[q][e] = 0.f;
          }
        }
#pragma unroll
        for (int blk = 0; blk < R::kPasses / R::kPassBlock; ++blk) {
          float sc[R::kPassBlock][kNQ];
          float mloc[kNQ];
#pragma unroll
          for (int q = 0; q < kNQ; ++q) mloc[q] = -INFINITY;
#pragma unroll
          for (int pb = 0; pb < R::kPassBlock; ++pb) {
            const int it = blk * R::kPassBlock + pb;
            const int r = warp * R::kKeysPerWarp + it * R::kRowsPerPass + grp;
            float f[EPL];
            load_slice<kBF16, R::kSliceBytes>(sK + r * R::kRowBytes + sub * R::kSliceBytes, f);
            if constexpr (kAppend) {
              if (r == subst) load_new_slice<kBF16, EPL>(knew_row, f);
            }
#pragma unroll
            for (int q = 0; q < kNQ; ++q) {
              float dot = 0.f;
#pragma unroll
              for (int e = 0; e < EPL; ++e) dot = fmaf(qv[q][e], f[e], dot);
#pragma unroll
              for (int off = LPR / 2; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
              sc[pb][q] = r < n ? dot : -INFINITY;
              mloc[q] = fmaxf(mloc[q], sc[pb][q]);
            }
          }
          float mnew[kNQ];
#pragma unroll
          for (int q = 0; q < kNQ; ++q) {
            mnew[q] = fmaxf(m[q], mloc[q]);
            const float corr = mnew[q] == -INFINITY ? 1.f : rescale(m[q], mnew[q]);
            ssum[q] *= corr;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[q][e] *= corr;
            m[q] = mnew[q];
          }
#pragma unroll
          for (int pb = 0; pb < R::kPassBlock; ++pb) {
            const int it = blk * R::kPassBlock + pb;
            const int r = warp * R::kKeysPerWarp + it * R::kRowsPerPass + grp;
            if (r < n) {
              float f[EPL];
              load_slice<kBF16, R::kSliceBytes>(sV + r * R::kRowBytes + sub * R::kSliceBytes, f);
              if constexpr (kAppend) {
                if (r == subst) load_new_slice<kBF16, EPL>(vnew_row, f);
              }
#pragma unroll
              for (int q = 0; q < kNQ; ++q) {
                const float pw = exp2f(sc[pb][q] - m[q]);
                ssum[q] += pw;
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[q][e] = fmaf(pw, f[e], acc[q][e]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[kStages + s]));

      const bool row_ends = seg_ends(cur, i);
      if (row_ends) {
        // ---- hand the row's state to the merge warp: merge this warp's lane groups,
        //      leave the warp's state in slot re & 1 and go on with the next chunk
        const int slot = re & 1;
        if (re >= 2 && !mbar_wait(smem_u32(&rbars[2 + slot]), static_cast<uint32_t>(((re >> 1) - 1) & 1), s_flags)) {
          ok = false;                                      // the merge warp has not read this slot
          s_flags[0] = 1;
          atomicOr(p.status, 1u);
        }
        float* sl_red = s_slots + slot * kSlotFloats;
        float* sl_m = sl_red + kNQ * kSlotWarps * kDh;
        float* sl_s = sl_m + kNQ * kSlotWarps;
        float* sl_ok = sl_s + kNQ * kSlotWarps;
#pragma unroll
        for (int q = 0; q < kNQ; ++q) {
#pragma unroll
          for (int off = LPR; off < 32; off <<= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[q], off);
            const float so = __shfl_xor_sync(0xffffffffu, ssum[q], off);
            const float M = fmaxf(m[q], mo);
            const float f0 = rescale(m[q], M), f1 = rescale(mo, M);
            ssum[q] = ssum[q] * f0 + so * f1;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
              const float ao = __shfl_xor_sync(0xffffffffu, acc[q][e], off);
              acc[q][e] = acc[q][e] * f0 + ao * f1;
            }
            m[q] = M;
          }
          if (lane < LPR) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) sl_red[(q * kSlotWarps + warp) * kDh + sub * EPL + e] = acc[q][e];
          }
          if (lane == 0) {
            sl_m[q * kSlotWarps + warp] = m[q];
            sl_s[q * kSlotWarps + warp] = ssum[q];
          }
        }
        if (lane == 0) sl_ok[warp] = ok ? 1.f : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&rbars[slot]));   // release: the slot's writes come first
        ++re;
#pragma unroll
        for (int q = 0; q < kNQ; ++q) {
          m[q] = -INFINITY;
          ssum[q] = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[q][e] = 0.f;
        }
      }
      const int prev_b = cur.b, prev_lh = cur.lh;
      step(cur, i);
      if (cur.b != prev_b || cur.lh != prev_lh) seg_c0 = cur.c;
    }
  }
  __syncthreads();
}

size_t counters_bytes(int B, int L, int H) {
  const size_t n = static_cast<size_t>(B) * L * H * sizeof(unsigned int);
  return (n + 255) & ~static_cast<size_t>(255);
}

template <bool kBF16, int kNQ, bool kAppend, bool kShallow = false>
size_t dynamic_smem_bytes(int B) {
  using R = Traits<kBF16, kNQ, kAppend, kShallow>;
  constexpr int kStages = R::kStages;
  size_t n = static_cast<size_t>(kStages) * R::kStageBytes;
  n += (2 * kStages + 4) * sizeof(uint64_t);
  n += static_cast<size_t>(B + 1) * sizeof(long long);
  n += static_cast<size_t>(B + (B & 1)) * sizeof(int);
  n += 2 * (static_cast<size_t>(kNQ) * R::kSlotWarps * (kDh + 2) + kConsumerWarps) * sizeof(float) + 4 * sizeof(int);
  if (R::kKeyLanes) n += 16 + static_cast<size_t>(R::kPFloats) * sizeof(float);
  return n;
}

template <bool kBF16, int kNQ, bool kAppend = false, bool kShallow = false>
cudaError_t launch(const DecodeParams& prm, const DeviceInfo& dev, cudaStream_t stream) {
  // per device: the largest shared memory set on the kernel so far, and the CTAs
  // per SM for the last shared-memory size queried (the host path stays cheap)
  static std::mutex mu;
  static size_t attr_bytes[128] = {};
  static size_t occ_bytes[128] = {};
  static int occ_ctas[128] = {};
  const size_t smem = dynamic_smem_bytes<kBF16, kNQ, kAppend, kShallow>(prm.B);
  constexpr int kCtas = min_ctas_per_sm<kBF16, kNQ, kAppend, kShallow>();
  cudaError_t e;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    const int d = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
    if (attr_bytes[d] < smem) {
      e = cudaFuncSetAttribute(decode_stream_kernel<kBF16, kNQ, kAppend, kShallow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_bytes[d] = smem;
    }
    if (occ_bytes[d] != smem) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_stream_kernel<kBF16, kNQ, kAppend, kShallow>, kThreads,
                                                        smem);
      if (e != cudaSuccess) return e;
      occ_bytes[d] = smem;
      occ_ctas[d] = per_sm;
    }
    per_sm = occ_ctas[d];
  }
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int grid = dev.num_sms * (per_sm < kCtas ? per_sm : kCtas);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = CXA_DECODE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_stream_kernel<kBF16, kNQ, kAppend, kShallow>, prm);
}

// One query per row: the deep ring, unless the stream is so long (an upper bound on
// its chunks from the host-side geometry; the key lengths live on the device) that
// launch tails matter little and more CTAs per SM stream faster.
constexpr long long kLongStreamChunks = 40960;
template <bool kBF16>
cudaError_t launch_one_query(const DecodeParams& prm, const DeviceInfo& dev, cudaStream_t stream) {
  using R = Traits<kBF16, 1>;
  const long long chunks = static_cast<long long>(prm.B) * prm.LH * ((prm.T + R::kChunkKeys - 1) / R::kChunkKeys);
  if (chunks >= kLongStreamChunks) return launch<kBF16, 1, false, true>(prm, dev, stream);
  return launch<kBF16, 1, false, false>(prm, dev, stream);
}

// fp32 cache: one instance per query-count bucket (a bf16 cache with several
// queries goes to the tensor-core kernel)
cudaError_t launch_f32_nq(const DecodeParams& prm, const DeviceInfo& dev, cudaStream_t stream) {
  if (prm.nq == 1) return launch_one_query<false>(prm, dev, stream);
  if (prm.nq == 2) return launch<false, 2>(prm, dev, stream);
  if (prm.nq <= 4) return launch<false, 4>(prm, dev, stream);
  if (prm.nq <= 6) return launch<false, 6>(prm, dev, stream);   // a beam of five or six
  return launch<false, 8>(prm, dev, stream);
}

}  // namespace

size_t decode_workspace_bytes(int B, int T, int L, int H, int nq) {
  const size_t nslot = static_cast<size_t>((T + kPartChunk - 1) / kPartChunk);
  return counters_bytes(B, L, H) + static_cast<size_t>(B) * L * H * nq * nslot * kPartFloats * sizeof(float);
}

size_t decode_counter_bytes(int B, int L, int H) { return counters_bytes(B, L, H); }

cudaError_t launch_decode(const DecodeLaunch& a, const DeviceInfo& dev, cudaStream_t stream,
                          std::string* msg) {
  // three or more queries per row of a bf16 cache: scores on the tensor cores
  // (bf16 x bf16 products are exact; an fp32 cache keeps fp32 scores here)
  if (a.nq >= 2 && a.cache_bf16) return launch_decode_shared_tc(a, dev, stream, msg);
  DecodeParams prm;
  prm.Q = a.Q;
  prm.Kc = static_cast<const uint8_t*>(a.Kc);
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
  prm.key_len_add = a.key_len_add;
  prm.part_stride = (a.T + kPartChunk - 1) / kPartChunk;
  prm.qscale = a.scale * 1.4426950408889634f;   // scale * log2(e)
  prm.Knew = a.K_new;
  prm.Vnew = a.V_new;
  cudaError_t e;
  if (a.nq == 1 && a.K_new == nullptr) {
    // short streams (a single memory or a few): the latency shape, a cluster per row
    if (decode_rows_eligible(a.B * a.nl * a.H, a.T, dev.num_sms, decode_policy())) {
      bool done = false;
      const cudaError_t er = launch_decode_rows(a, dev, stream, &done);
      if (er != cudaSuccess || done) return er;
    }
  }
  if (a.K_new != nullptr)   // the self-attention step: append fused into a one-query decode
    e = a.cache_bf16 ? launch<true, 1, true>(prm, dev, stream) : launch<false, 1, true>(prm, dev, stream);
  else
    e = a.cache_bf16 ? launch_one_query<true>(prm, dev, stream) : launch_f32_nq(prm, dev, stream);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace cxa
