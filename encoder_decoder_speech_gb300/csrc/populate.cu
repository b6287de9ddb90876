// Populate: K_l = E x WK_l and V_l = E x WV_l + bV_l for every decoder layer at
// once, written directly into the layer-major, head-major cache.
//
// ("Whisper: Trace One Encoder Tensor into Every Decoder Layer": "The concept"
// gives the per-layer projections of the one encoder memory; "Deliberate
// failure" the token-major -> head-major re-layout that the GEMM epilogue here
// performs in place of a separate transpose pass; "View 2" the per-layer slab.)
//
// All L layers' K and V projections form one GEMM per encoder memory:
//   C[t, n] = sum_i E[t, i] * Wcat[i, n],   n = (kv*L + l)*d + h*64 + c
// with M = T rows per slot, N = 2*L*d, K = d. Two kernels:
//   1. pack_weights: WK/WV [L][d_in][d_out] -> Wp [2*L*d][d] (K-major, the
//      operand layout the tensor core reads without a transpose flag). The
//      weights are static across audio windows ("The concept": only E changes),
//      so a caller packs them once (cxa_pack_weights) and populates every later
//      window from the packed copy (cxa_populate_packed); cxa_populate does both.
//   2. populate_gemm: persistent, warp-specialised tcgen05 GEMM.
//        warp 0     TMA producer (one thread): E tile 128 x 128 B and Wp tile
//                   256 x 128 B per k-block, 128-byte swizzled, 4-stage ring.
//        warp 1     TMEM allocator + MMA issuer (one thread): 128x256 fp32
//                   accumulator, two accumulators in TMEM (512 columns) so the
//                   epilogue of one tile overlaps the main loop of the next.
//        warps 2-5  epilogue: tcgen05.ld rows out of TMEM, add bV on V columns,
//                   optionally round to bf16, stage 128-row boxes in shared
//                   memory and write each to Kc/Vc[b][l][h][t][:] with one bulk
//                   tensor store.
//      For large GEMMs the same kernel runs on CTA pairs (clusters of two,
//      tcgen05 cta_group::2): a 256 x 256 tile per pair, each CTA loading its 128
//      rows of E and 128 of the tile's 256 weight rows per k-block (6-stage ring
//      of 32 KB stages), the even CTA issuing the MMAs for both and signalling
//      both CTAs' barriers, each CTA draining its own 128 accumulator rows.
//      Tiles never straddle two encoder memories (M tiles are per slot; rows
//      t >= T are zero-filled by TMA and never stored).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>
#include <type_traits>

#include "cxa.h"
#include "internal.h"
#include "chunk_stream.cuh"
#include "cluster.cuh"
#include "ptx.cuh"

namespace cxa {
namespace {

constexpr int kBM = 128;                       // rows (tokens) per CTA and tile = TMEM lanes
constexpr int kBN = 256;                       // columns per tile = 4 heads of 64
constexpr uint32_t kRowBytes = 128;            // one k-block row: 32 fp32 / 64 bf16
constexpr uint32_t kABytes = kBM * kRowBytes;  // 16 KB
constexpr uint32_t kTmemCols = 2 * kBN;        // two accumulators
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr uint32_t kBoxBytes = kBM * 128;      // one store box: the tile's 128 rows x 128 bytes
constexpr uint32_t kStagingBytes = 2 * kBoxBytes;   // double-buffered, shared by the epilogue warps
constexpr int kEpiBarrier = 1;                 // named barrier of the 4 epilogue warps

// One CTA per tile (kPair false: a 128 x 256 tile, 4-stage ring of 48 KB stages), or
// a CTA pair per tile (kPair true: cta_group::2, a 256 x 256 tile whose A rows and B
// rows are split between the two CTAs, so each stage holds 16 KB of A and 16 KB of
// B and the ring is 6 deep).
template <bool kPair>
struct Shape {
  static constexpr int kStages = kPair ? 6 : 4;
  static constexpr int kTileM = kPair ? 2 * kBM : kBM;          // rows per tile
  static constexpr uint32_t kBRows = kPair ? kBN / 2 : kBN;     // B rows one CTA loads
  static constexpr uint32_t kBBytes = kBRows * kRowBytes;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kNumBarriers = 2 * kStages + 4 + 1;
  static constexpr size_t kSmemBytes =
      1024 + size_t(kStages) * kStageBytes + kStagingBytes + 8 * kNumBarriers + 16;
  static_assert(kSmemBytes + 16 <= 227 * 1024, "dynamic + static shared memory fits one CTA");
};

struct GemmParams {
  void* Kc;
  void* Vc;
  const float* bV;
  unsigned int* status;
  int b0, T, d, L, H;
  int mt_per_slot;     // ceil(T / 128)
  int num_m_tiles;     // nb * mt_per_slot
  int num_tiles;       // num_m_tiles * num_n_tiles
  int raster_n;        // 1: consecutive tiles walk N under one M tile (E rows reused), 0: walk M
  int num_kb;          // d / k-block elements
  int num_heads_total; // 2 * L * H
  int cache_bf16;
};

__device__ __forceinline__ void report_timeout(unsigned int* status, volatile int* abort) {
  *abort = 1;
  atomicOr(status, 1u);
}

template <bool kBF16In, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    populate_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const GemmParams p) {
  using S = Shape<kPair>;
  constexpr int kStages = S::kStages;
  constexpr int kNumBarriers = S::kNumBarriers;
  constexpr uint32_t kBBytes = S::kBBytes;
  constexpr uint32_t kStageBytes = S::kStageBytes;
  constexpr int kKElems = kBF16In ? 64 : 32;   // elements per 128-byte k-block row
  constexpr int kKStep = kBF16In ? 16 : 8;     // K of one MMA instruction
  constexpr int kMmasPerBlock = kKElems / kKStep;
  constexpr uint32_t kStepBytes = kKStep * (kBF16In ? 2 : 4);   // 32 bytes

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + kStages * kABytes;
  const uint32_t staging = base + kStages * kStageBytes;   // 1024-byte aligned
  const uint32_t bars = staging + kStagingBytes;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto tfull_bar = [&](int a) { return bars + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bars + 8u * (2 * kStages + 2 + a); };
  const uint32_t drain_bar = bars + 8u * (2 * kStages + 4);
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(base_ptr + kStages * kStageBytes + kStagingBytes + 8 * kNumBarriers);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A pair: rank 0 (the even CTA) issues the MMAs and owns the full and accumulator-
  // empty barriers both CTAs count on; rank 1 loads and drains its halves.
  const uint32_t rank = kPair ? cluster_rank() : 0u;
  const bool even = rank == 0;
  const int tile0 = kPair ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int tile_step = kPair ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kPair ? 2 * kEpiWarps : kEpiWarps);   // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (kPair)
    cluster_sync();   // both CTAs' barriers are initialised before any cross-CTA arrival
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < p.num_tiles; tile += tile_step) {
        const int mtg = p.raster_n ? tile / (p.num_tiles / p.num_m_tiles) : tile % p.num_m_tiles;
        const int nt = p.raster_n ? tile % (p.num_tiles / p.num_m_tiles) : tile / p.num_m_tiles;
        const int slot = mtg / p.mt_per_slot;
        const int mt = mtg - slot * p.mt_per_slot;
        const int row0 = mt * S::kTileM + static_cast<int>(rank) * kBM;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if constexpr (kPair) {
            // both halves complete on the even CTA's full barrier, which expects them both
            if (even) mbar_arrive_expect_tx(full_bar(stage), 2 * kStageBytes);
            const uint32_t fb = mapa_shared(full_bar(stage), 0);
            tma_load_3d_pair(sA + stage * kABytes, &tmA, fb, kb * kKElems, row0, slot);
            tma_load_2d_pair(sB + stage * kBBytes, &tmB, fb, kb * kKElems,
                             nt * kBN + static_cast<int>(rank * S::kBRows));
          } else {
            mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
            tma_load_3d(sA + stage * kABytes, &tmA, full_bar(stage), kb * kKElems, row0, slot);
            tma_load_2d(sB + stage * kBBytes, &tmB, full_bar(stage), kb * kKElems, nt * kBN);
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        report_timeout(p.status, abort_flag);
        // Let every copy already issued land before the CTA can exit (a pair's copies
        // complete on the even CTA's barriers; the odd CTA then stays until the final
        // cluster barrier, which the even CTA reaches after these waits).
        if (!kPair || even)
          for (int s = 0; s < kStages; ++s)
            if (armed & (1u << s)) mbar_wait(full_bar(s), (armed_parity >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && even) {
      constexpr uint32_t idesc = make_idesc(kBF16In ? 1u : 2u, S::kTileM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < p.num_tiles; tile += tile_step) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sA + stage * kABytes;
          const uint32_t b0 = sB + stage * kBBytes;
#pragma unroll
          for (int k = 0; k < kMmasPerBlock; ++k) {
            const uint64_t ad = smem_desc_k_sw128(a0 + k * kStepBytes);
            const uint64_t bd = smem_desc_k_sw128(b0 + k * kStepBytes);
            const uint32_t accumulate = (kb | k) != 0 ? 1u : 0u;
            if constexpr (kPair) {
              if constexpr (kBF16In)
                mma_bf16_pair(d_tmem, ad, bd, idesc, accumulate);
              else
                mma_tf32_pair(d_tmem, ad, bd, idesc, accumulate);
            } else {
              if constexpr (kBF16In)
                mma_bf16(d_tmem, ad, bd, idesc, accumulate);
              else
                mma_tf32(d_tmem, ad, bd, idesc, accumulate);
            }
          }
          // frees the smem stage (of both CTAs) once these MMAs finish
          if constexpr (kPair)
            tc_commit_pair(empty_bar(stage), 0x3);
          else
            tc_commit(empty_bar(stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator ready for the epilogue (of both CTAs)
        if constexpr (kPair)
          tc_commit_pair(tfull_bar(acc), 0x3);
        else
          tc_commit(tfull_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) report_timeout(p.status, abort_flag);
      // Every MMA issued must complete before TMEM is released.
      if constexpr (kPair)
        tc_commit_pair(drain_bar, 0x1);
      else
        tc_commit(drain_bar);
      if (!mbar_wait(drain_bar, 0)) report_timeout(p.status, abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Each warp owns TMEM lanes 32*quad .. 32*quad+31 = 32 consecutive tokens t of
    // one memory. For every 64-column head block the four warps read their
    // accumulator rows, add bV on V columns and write them into one 128-row box of
    // 128 bytes per row in shared memory (128-byte swizzle, conflict-free: the
    // 16-byte chunk j of row r lands at slot j ^ (r & 7), the layout the cache's
    // tensor maps read); one thread then writes the box into the head-major cache,
    // where the tile's rows t are contiguous, with one bulk tensor store (rows
    // t >= T lie outside the map and are not written). A tile goes out as 8 boxes
    // (fp32 cache) or 4 (bf16). With CTA pairs this measured 2-10 % faster than
    // 16-byte stores from all 128 threads (the one-CTA kernel on a single fp32 tile
    // per CTA, Whisper-tiny dims, ~0.4 us slower).
    const int quad = warp & 3;
    const bool leader = warp == 2 && lane == 0;  // reads the abort flag and issues the bulk stores
    const int LH = p.L * p.H;
    const uint32_t swz = static_cast<uint32_t>(lane & 7);
    int acc = 0;
    uint32_t acc_phase = 0;
    int sbuf = 0;
    // one box: write this warp's 32 rows into the staging buffer, then one thread
    // stores the box. The buffer alternates, so one barrier per box suffices: before
    // that barrier the storing thread waits until the previous box's bulk store has
    // read its buffer, which the next box rewrites after the barrier.
    auto put_box = [&](const uint32_t (&w)[8][4], const CUtensorMap* tm, int c0, int t0, int row3) {
      const uint32_t buf = staging + static_cast<uint32_t>(sbuf) * kBoxBytes;
      const uint32_t mine = buf + static_cast<uint32_t>(quad * 32 + lane) * 128u;
#pragma unroll
      for (int j = 0; j < 8; ++j) st_shared_v4(mine + ((static_cast<uint32_t>(j) ^ swz) << 4), w[j][0], w[j][1], w[j][2], w[j][3]);
      fence_proxy_async_smem();                                 // the box, before the bulk store reads it
      if (leader) bulk_wait_group_read<0>();                    // the previous box's store has read its buffer
      named_barrier(kEpiBarrier, kEpiWarps * 32);               // every row is written
      if (leader && t0 < p.T) {                                  // a box wholly past T is not stored at all
        tma_store_3d(tm, buf, c0, t0, row3);                    // rows t >= T lie outside the map: not written
        bulk_commit_group();
      }
      sbuf ^= 1;
    };
    __shared__ int s_epi_stop;
    for (int tile = tile0; tile < p.num_tiles; tile += tile_step) {
      // The four warps must take the same path through the tile (named barriers):
      // each reports its own wait's timeout, then one thread reads the abort flag
      // once for all of them.
      const bool got = mbar_wait(tfull_bar(acc), acc_phase, abort_flag);
      if (!got && lane == 0) report_timeout(p.status, abort_flag);
      named_barrier(kEpiBarrier, kEpiWarps * 32);
      if (leader) s_epi_stop = *abort_flag;
      named_barrier(kEpiBarrier, kEpiWarps * 32);
      if (s_epi_stop != 0) break;
      tc_fence_after();
      const int mtg = p.raster_n ? tile / (p.num_tiles / p.num_m_tiles) : tile % p.num_m_tiles;
      const int nt = p.raster_n ? tile % (p.num_tiles / p.num_m_tiles) : tile / p.num_m_tiles;
      const int slot = mtg / p.mt_per_slot;
      const int mt = mtg - slot * p.mt_per_slot;
      const int t0 = mt * S::kTileM + static_cast<int>(rank) * kBM;   // first token of this CTA's rows
      const int b = p.b0 + slot;
#pragma unroll 1
      for (int g = 0; g < kBN / 64; ++g) {
        const int head = nt * (kBN / 64) + g;
        if (head >= p.num_heads_total) break;
        const int kv = head / LH;
        const int lh = head - kv * LH;
        const int l = lh / p.H;
        const int h = lh - l * p.H;
        const int row3 = b * LH + lh;
        uint32_t r[2][32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                 static_cast<uint32_t>(acc * kBN + g * 64 + half * 32);
          tmem_ld_32x32b_x32(taddr, r[half]);
        }
        tmem_ld_wait();
        if (kv) {
          const float4* bv4 = reinterpret_cast<const float4*>(p.bV + static_cast<size_t>(l) * p.d + h * 64);
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 bb = __ldg(bv4 + half * 8 + i);
              r[half][4 * i + 0] = __float_as_uint(__uint_as_float(r[half][4 * i + 0]) + bb.x);
              r[half][4 * i + 1] = __float_as_uint(__uint_as_float(r[half][4 * i + 1]) + bb.y);
              r[half][4 * i + 2] = __float_as_uint(__uint_as_float(r[half][4 * i + 2]) + bb.z);
              r[half][4 * i + 3] = __float_as_uint(__uint_as_float(r[half][4 * i + 3]) + bb.w);
            }
        }
        if (p.cache_bf16) {
          // one box: 64 bf16 channels = 128 bytes per row
          uint32_t w[8][4];
#pragma unroll
          for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int c = 8 * j + 2 * k;      // channels c, c+1
              __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(r[c >> 5][c & 31]),
                                                        __uint_as_float(r[(c + 1) >> 5][(c + 1) & 31]));
              w[j][k] = *reinterpret_cast<uint32_t*>(&pr);
            }
          put_box(w, kv ? &tmV : &tmK, 0, t0, row3);
        } else {
          // two boxes: channels 0-31 and 32-63, 128 bytes of fp32 per row each
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t w[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
              for (int k = 0; k < 4; ++k) w[j][k] = r[half][4 * j + k];
            put_box(w, kv ? &tmV : &tmK, half * 32, t0, row3);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair)
          mbar_arrive_cluster(tempty_bar(acc), 0);   // the even CTA's MMA waits for both CTAs
        else
          mbar_arrive(tempty_bar(acc));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (leader) bulk_wait_group_all();   // every bulk store complete before the CTA leaves
    __syncwarp();
  }

  tc_fence_before();
  if constexpr (kPair)
    cluster_sync();   // neither CTA leaves while the pair's MMAs or arrivals may still touch it
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// WK/WV [L][d_in][d_out] -> Wp[(kv*L + l)*d + j][i] (K-major). fp32 weights are
// rounded to TF32 (round to nearest, ties away from zero: cvt.rna.tf32.f32).
// One 64 x 64 tile per CTA: 16-byte global loads along d_out, a transposed
// shared-memory tile whose 16-byte chunks are XOR-swizzled so that neither the
// scattered writes nor the row reads conflict on banks, 16-byte global stores
// along d_in.
constexpr int kPackTile = 64;
constexpr int kPackThreads = 256;

template <bool kBF16In>
__global__ void __launch_bounds__(kPackThreads)
    pack_weights_kernel(const void* __restrict__ WK, const void* __restrict__ WV,
                        void* __restrict__ Wp, int d, int L) {
  using Elem = typename std::conditional<kBF16In, uint16_t, uint32_t>::type;
  constexpr int V = 16 / sizeof(Elem);              // elements per 16-byte chunk
  constexpr int kChunks = kPackTile / V;            // chunks per tile row
  __shared__ __align__(16) Elem tile[kPackTile][kPackTile];   // tile[j][i], chunk-swizzled

  const int kvl = blockIdx.z;
  const int kv = kvl / L;
  const int l = kvl - kv * L;
  const Elem* W = static_cast<const Elem*>(kv ? WV : WK) + static_cast<size_t>(l) * d * d;
  Elem* out = static_cast<Elem*>(Wp);
  const int i0 = blockIdx.y * kPackTile;            // d_in
  const int j0 = blockIdx.x * kPackTile;            // d_out

  for (int idx = threadIdx.x; idx < kPackTile * kChunks; idx += kPackThreads) {
    const int r = idx / kChunks;                    // d_in row of the source tile
    const int cv = idx - r * kChunks;               // 16-byte chunk along d_out
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(W + static_cast<size_t>(i0 + r) * d + j0 + cv * V));
    const Elem* e = reinterpret_cast<const Elem*>(&u);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int j = cv * V + k;                     // transposed row
      const int chunk = (r / V) ^ ((j / V) & 7);
      tile[j][chunk * V + (r % V)] = e[k];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kPackTile * kChunks; idx += kPackThreads) {
    const int j = idx / kChunks;                    // d_out row of the packed tile
    const int q = idx - j * kChunks;                // 16-byte chunk along d_in
    uint4 u = *reinterpret_cast<const uint4*>(&tile[j][(q ^ ((j / V) & 7)) * V]);
    if constexpr (!kBF16In) {
      uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(w[k]) : "f"(__uint_as_float(w[k])));
    }
    *reinterpret_cast<uint4*>(out + (static_cast<size_t>(kvl) * d + j0 + j) * d + i0 + q * V) = u;
  }
}

// fp32 -> bf16, round to nearest even: the conversion pass in front of the bf16
// populate when the encoder memory (or a weight) arrives in fp32. Each thread
// turns 8 values (two 16-byte loads) into one 16-byte store; the ragged tail of
// n % 8 values is done one by one. HBM-bound: 6 bytes moved per value.
constexpr int kConvertThreads = 256;

__global__ void __launch_bounds__(kConvertThreads)
    convert_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, size_t n) {
  const size_t groups = n / 8;
  const size_t stride = static_cast<size_t>(gridDim.x) * kConvertThreads;
  for (size_t g = static_cast<size_t>(blockIdx.x) * kConvertThreads + threadIdx.x; g < groups; g += stride) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(src) + 2 * g);
    const float4 b = __ldcs(reinterpret_cast<const float4*>(src) + 2 * g + 1);
    __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
    reinterpret_cast<uint4*>(dst)[g] =
        make_uint4(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1),
                   *reinterpret_cast<uint32_t*>(&p2), *reinterpret_cast<uint32_t*>(&p3));
  }
  if (blockIdx.x == 0 && threadIdx.x < n % 8) {
    const size_t i = groups * 8 + threadIdx.x;
    dst[i] = __float2bfloat16_rn(src[i]);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder(std::string* msg) {
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
  if (fn == nullptr) *msg = "cuTensorMapEncodeTiled is not available from the CUDA driver";
  return fn;
}

template <bool kBF16In, bool kPair>
cudaError_t set_smem_attr_once(int device) {
  static std::mutex mu;
  static bool done[128] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 128 && done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(populate_gemm_kernel<kBF16In, kPair>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Shape<kPair>::kSmemBytes));
  if (e == cudaSuccess && device >= 0 && device < 128) done[device] = true;
  return e;
}

// CTA pairs of the pair kernel resident on the device at once (queried once per
// device and input dtype), or -1 when pairs cannot be launched.
template <bool kBF16In>
int pair_clusters(const DeviceInfo& dev) {
  static std::mutex mu;
  static int cache[128] = {};
  const int dv = dev.device >= 0 && dev.device < 128 ? dev.device : 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dv] != 0) return cache[dv];
  }
  int n = 0;
  if (set_smem_attr_once<kBF16In, true>(dev.device) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Shape<true>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, populate_gemm_kernel<kBF16In, true>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  cache[dv] = n > 0 ? n : -1;
  return cache[dv];
}

template <bool kBF16In>
cudaError_t run(const PopulateLaunch& a, const DeviceInfo& dev, cudaStream_t stream, std::string* msg) {
  const int esz = kBF16In ? 2 : 4;
  const int kKElems = 128 / esz;
  const int N = 2 * a.L * a.d;

  // 1. tensor maps: E as (d, T, nb), Wp (the packed weights) as (d, N); 128-byte
  //    rows, 128-byte swizzle
  EncodeTiledFn encode = tensor_map_encoder(msg);
  if (encode == nullptr) return cudaErrorInvalidValue;
  const CUtensorMapDataType dt = kBF16In ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  // CTA pairs (cta_group::2) when the policy asks for them, or under the automatic
  // choice when pairs can be resident and the GEMM spans at least four waves of
  // one-CTA tiles (measured on GB300: below that the pairs' 256-row tiles leave more
  // SMs idle in the last wave than the halved operand loads save); one CTA per tile
  // otherwise
  const int policy = populate_policy();
  const long long single_tiles = static_cast<long long>(a.nb) * ((a.T + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  const bool want_pair = policy == CXA_POPULATE_PAIR ||
                         (policy == CXA_POPULATE_AUTO && single_tiles >= 4LL * dev.num_sms);
  const int pairs = want_pair ? pair_clusters<kBF16In>(dev) : 0;
  if (policy == CXA_POPULATE_PAIR && pairs <= 0) {
    *msg = "CTA pairs of the populate kernel cannot be resident on this device (policy CXA_POPULATE_PAIR)";
    return cudaErrorInvalidValue;
  }
  const bool pair = pairs > 0;
  const int tile_m = pair ? Shape<true>::kTileM : Shape<false>::kTileM;
  const uint32_t b_rows = pair ? Shape<true>::kBRows : Shape<false>::kBRows;
  CUtensorMap tmA, tmB;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.d), static_cast<cuuint64_t>(a.T), static_cast<cuuint64_t>(a.nb)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.d) * esz, static_cast<cuuint64_t>(a.T) * a.d * esz};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kKElems), static_cast<cuuint32_t>(kBM), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(&tmA, dt, 3, const_cast<void*>(a.E), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *msg = "cuTensorMapEncodeTiled failed for E (code " + std::to_string(static_cast<int>(r)) + ")";
      return cudaErrorInvalidValue;
    }
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.d), static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.d) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kKElems), static_cast<cuuint32_t>(b_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&tmB, dt, 2, const_cast<void*>(a.wpack), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *msg = "cuTensorMapEncodeTiled failed for the packed weights (code " + std::to_string(static_cast<int>(r)) + ")";
      return cudaErrorInvalidValue;
    }
  }

  // the cache as (64 channels, T, B*L*H rows) for the epilogue's bulk stores: a box is the
  // tile's 128 rows of 128 bytes (32 fp32 / 64 bf16 channels)
  CUtensorMap tmK, tmV;
  {
    const CUtensorMapDataType ct = a.cache_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int ces = a.cache_bf16 ? 2 : 4;
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(a.T), static_cast<cuuint64_t>(a.B) * a.L * a.H};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(64 * ces), static_cast<cuuint64_t>(a.T) * 64 * ces};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / ces), static_cast<cuuint32_t>(kBM), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    for (int kv = 0; kv < 2; ++kv) {
      CUresult r = encode(kv ? &tmV : &tmK, ct, 3, kv ? a.Vc : a.Kc, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) {
        *msg = "cuTensorMapEncodeTiled failed for the cache (code " + std::to_string(static_cast<int>(r)) + ")";
        return cudaErrorInvalidValue;
      }
    }
  }
  cudaError_t e = pair ? set_smem_attr_once<kBF16In, true>(dev.device) : set_smem_attr_once<kBF16In, false>(dev.device);
  if (e != cudaSuccess) return e;

  // 2. the persistent GEMM over the packed weights
  GemmParams p;
  p.Kc = a.Kc;
  p.Vc = a.Vc;
  p.bV = a.bV;
  p.status = dev.status_word;
  p.b0 = a.b0;
  p.T = a.T;
  p.d = a.d;
  p.L = a.L;
  p.H = a.H;
  p.mt_per_slot = (a.T + tile_m - 1) / tile_m;
  p.num_m_tiles = a.nb * p.mt_per_slot;
  const int num_n_tiles = (N + kBN - 1) / kBN;
  p.num_tiles = p.num_m_tiles * num_n_tiles;
  // Walk N under one M tile when all packed weights stay in L2 while the cache writes
  // stream past (E rows are then read once); otherwise walk M, so that each wave
  // shares one weight tile and E (the smaller operand) is what L2 holds.
  const size_t w_bytes = static_cast<size_t>(N) * a.d * (kBF16In ? 2 : 4);
  p.raster_n = w_bytes <= (32u << 20) ? 1 : 0;
  p.num_kb = a.d / kKElems;
  p.num_heads_total = 2 * a.L * a.H;
  p.cache_bf16 = a.cache_bf16 ? 1 : 0;


  if (pair) {
    const int clusters = p.num_tiles < pairs ? p.num_tiles : pairs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Shape<true>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, populate_gemm_kernel<kBF16In, true>, tmA, tmB, tmK, tmV, p);
  } else {
    const int grid = p.num_tiles < dev.num_sms ? p.num_tiles : dev.num_sms;
    populate_gemm_kernel<kBF16In, false><<<grid, kThreads, Shape<false>::kSmemBytes, stream>>>(tmA, tmB, tmK, tmV, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaSuccess;
}

}  // namespace

size_t populate_workspace_bytes(int d, int L, bool in_bf16) {
  return static_cast<size_t>(2) * L * d * d * (in_bf16 ? 2 : 4);
}

cudaError_t launch_populate(const PopulateLaunch& a, const DeviceInfo& dev, cudaStream_t stream,
                            std::string* msg) {
  return a.in_bf16 ? run<true>(a, dev, stream, msg) : run<false>(a, dev, stream, msg);
}

cudaError_t launch_convert_bf16(const float* src, void* dst, size_t n, const DeviceInfo& dev, cudaStream_t stream) {
  const size_t groups = n / 8;
  size_t grid = (groups + kConvertThreads - 1) / kConvertThreads;
  const size_t cap = static_cast<size_t>(dev.num_sms) * 8;   // 8 resident CTAs of 256 threads per SM
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  convert_bf16_kernel<<<static_cast<unsigned int>(grid), kConvertThreads, 0, stream>>>(
      src, static_cast<__nv_bfloat16*>(dst), n);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

cudaError_t launch_pack_weights(const void* WK, const void* WV, void* wpack, int d, int L, bool in_bf16,
                                cudaStream_t stream) {
  const dim3 grid(d / kPackTile, d / kPackTile, 2 * L);
  if (in_bf16)
    pack_weights_kernel<true><<<grid, kPackThreads, 0, stream>>>(WK, WV, wpack, d, L);
  else
    pack_weights_kernel<false><<<grid, kPackThreads, 0, stream>>>(WK, WV, wpack, d, L);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace cxa
