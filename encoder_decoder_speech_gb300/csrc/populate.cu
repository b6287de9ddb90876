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
//                   memory and write them with coalesced 16-byte stores to
//                   Kc/Vc[b][l][h][t][:].
//      Tiles never straddle two encoder memories (M tiles are per slot; rows
//      t >= T are zero-filled by TMA and never stored).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>
#include <type_traits>

#include "internal.h"
#include "chunk_stream.cuh"
#include "ptx.cuh"

namespace cxa {
namespace {

constexpr int kBM = 128;                       // rows (tokens) per tile = TMEM lanes
constexpr int kBN = 256;                       // columns per tile = 4 heads of 64
constexpr int kStages = 4;
constexpr uint32_t kRowBytes = 128;            // one k-block row: 32 fp32 / 64 bf16
constexpr uint32_t kABytes = kBM * kRowBytes;  // 16 KB
constexpr uint32_t kBBytes = kBN * kRowBytes;  // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 2 * kBN;        // two accumulators
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr uint32_t kBoxBytes = kBM * 128;      // one store box: the tile's 128 rows x 128 bytes
constexpr uint32_t kStagingBytes = 2 * kBoxBytes;   // double-buffered, shared by the epilogue warps
constexpr int kEpiBarrier = 1;                 // named barrier of the 4 epilogue warps
constexpr int kNumBarriers = 2 * kStages + 4 + 1;
constexpr size_t kSmemBytes =
    1024 + size_t(kStages) * kStageBytes + kStagingBytes + 8 * kNumBarriers + 16;

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

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

__device__ __forceinline__ void report_timeout(unsigned int* status, volatile int* abort) {
  *abort = 1;
  atomicOr(status, 1u);
}

template <bool kBF16In>
__global__ void __launch_bounds__(kThreads, 1)
    populate_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const GemmParams p) {
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);   // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
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
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int mtg = p.raster_n ? tile / (p.num_tiles / p.num_m_tiles) : tile % p.num_m_tiles;
        const int nt = p.raster_n ? tile % (p.num_tiles / p.num_m_tiles) : tile / p.num_m_tiles;
        const int slot = mtg / p.mt_per_slot;
        const int mt = mtg - slot * p.mt_per_slot;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
          tma_load_3d(sA + stage * kABytes, &tmA, full_bar(stage), kb * kKElems, mt * kBM, slot);
          tma_load_2d(sB + stage * kBBytes, &tmB, full_bar(stage), kb * kKElems, nt * kBN);
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
        // Let every copy already issued land before the CTA can exit.
        for (int s = 0; s < kStages; ++s)
          if (armed & (1u << s)) mbar_wait(full_bar(s), (armed_parity >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kBF16In ? 1u : 2u, kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
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
            if constexpr (kBF16In)
              mma_bf16(d_tmem, ad, bd, idesc, accumulate);
            else
              mma_tf32(d_tmem, ad, bd, idesc, accumulate);
          }
          tc_commit(empty_bar(stage));   // frees the smem stage once these MMAs finish
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));       // accumulator ready for the epilogue
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) report_timeout(p.status, abort_flag);
      // Every MMA issued must complete before TMEM is released.
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
    // 16-byte chunk j of row r lands at slot j ^ (r & 7)); the 128 threads then
    // read the box back in row order and write it with 16-byte stores into the
    // head-major cache, where the tile's rows t are contiguous; rows t >= T are
    // skipped. A tile goes out as 8 boxes (fp32 cache) or 4 (bf16). Storing the
    // boxes with TMA instead (first a box per warp, then a box per CTA) was slower.
    const int quad = warp & 3;
    const bool leader = warp == 2 && lane == 0;  // reads the abort flag for the epilogue
    const uint32_t ces = p.cache_bf16 ? 2u : 4u; // cache element bytes
    const int LH = p.L * p.H;
    const uint32_t swz = static_cast<uint32_t>(lane & 7);
    int acc = 0;
    uint32_t acc_phase = 0;
    int sbuf = 0;
    // one box: write this warp's 32 rows into the staging buffer, then all 128
    // threads read the box back in row order and store it with 16-byte global
    // stores (a warp writes four whole 128-byte rows per instruction); rows t >= T
    // are skipped. The buffer alternates, so one barrier per box suffices: a
    // buffer is rewritten two boxes later, after every thread has passed the
    // barrier that follows its last read of it.
    auto put_box = [&](const uint32_t (&w)[8][4], uint8_t* cache, int c0, int t0, int row3) {
      const uint32_t buf = staging + static_cast<uint32_t>(sbuf) * kBoxBytes;
      const uint32_t mine = buf + static_cast<uint32_t>(quad * 32 + lane) * 128u;
#pragma unroll
      for (int j = 0; j < 8; ++j) st_shared_v4(mine + ((static_cast<uint32_t>(j) ^ swz) << 4), w[j][0], w[j][1], w[j][2], w[j][3]);
      named_barrier(kEpiBarrier, kEpiWarps * 32);             // every row is written
      const int et = (warp - 2) * 32 + lane;                  // epilogue thread 0..127
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int q = et + m * kEpiWarps * 32;                // 16-byte chunk q of the box
        const int row = q >> 3, j = q & 7;
        if (t0 + row < p.T) {
          uint32_t v0, v1, v2, v3;
          ld_shared_v4(buf + static_cast<uint32_t>(row) * 128u + ((static_cast<uint32_t>(j ^ (row & 7))) << 4), v0, v1, v2, v3);
          uint8_t* dst = cache + (static_cast<size_t>(row3) * p.T + (t0 + row)) * (64u * ces) + c0 * ces + j * 16;
          *reinterpret_cast<uint4*>(dst) = make_uint4(v0, v1, v2, v3);
        }
      }
      sbuf ^= 1;
    };
    __shared__ int s_epi_stop;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
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
      const int t0 = mt * kBM;                  // first token of the tile
      const int b = p.b0 + slot;
#pragma unroll 1
      for (int g = 0; g < kBN / 64; ++g) {
        const int head = nt * (kBN / 64) + g;
        if (head >= p.num_heads_total) break;
        const int kv = head / LH;
        const int lh = head - kv * LH;
        const int l = lh / p.H;
        const int h = lh - l * p.H;
        uint8_t* cache = static_cast<uint8_t*>(kv ? p.Vc : p.Kc);
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
          put_box(w, cache, 0, t0, row3);
        } else {
          // two boxes: channels 0-31 and 32-63, 128 bytes of fp32 per row each
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t w[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
              for (int k = 0; k < 4; ++k) w[j][k] = r[half][4 * j + k];
            put_box(w, cache, half * 32, t0, row3);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
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

template <bool kBF16In>
cudaError_t set_smem_attr_once(int device) {
  static std::mutex mu;
  static bool done[128] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 128 && done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(populate_gemm_kernel<kBF16In>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e == cudaSuccess && device >= 0 && device < 128) done[device] = true;
  return e;
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
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kKElems), static_cast<cuuint32_t>(kBN)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&tmB, dt, 2, const_cast<void*>(a.wpack), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *msg = "cuTensorMapEncodeTiled failed for the packed weights (code " + std::to_string(static_cast<int>(r)) + ")";
      return cudaErrorInvalidValue;
    }
  }

  cudaError_t e = set_smem_attr_once<kBF16In>(dev.device);
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
  p.mt_per_slot = (a.T + kBM - 1) / kBM;
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

  const int grid = p.num_tiles < dev.num_sms ? p.num_tiles : dev.num_sms;
  populate_gemm_kernel<kBF16In><<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, p);
  e = cudaGetLastError();
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
