// Appending one row per (slot, layer, head) to a K/V cache: the self-attention
// KV cache of a decoder step, where each step writes the new token's key and
// value at position pos[b] and attends positions 0 .. pos[b] ("Caso de
// estudio: WhisperKit", §4: a fixed max_seq_len cache updated by a one-hot
// masked blend at the current position; "Recurrence as feeds", "What it
// opened": the new rows are written with scatter, the cache being an input and
// an output of the step).
//
// The masked blend cache*(1 - onehot(pos)) + new*onehot(pos) equals a scatter of
// the new row to position pos; here each row is one 16-lane store of 64 values.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "internal.h"

namespace cxa {
namespace {

constexpr int kAppendThreads = 256;   // 16 rows of 64 values per CTA (16 lanes x float4)

__global__ void __launch_bounds__(kAppendThreads)
    append_rows_kernel(const int* __restrict__ pos, const float* __restrict__ Knew, const float* __restrict__ Vnew,
                       void* Kc, void* Vc, int B, int LH, int T, int cache_bf16) {
  const long long row = static_cast<long long>(blockIdx.x) * (kAppendThreads / 16) + threadIdx.x / 16;
  const int lane16 = threadIdx.x % 16;
  if (row >= static_cast<long long>(B) * LH) return;
  const int b = static_cast<int>(row / LH);
  const int t = __ldg(pos + b);
  if (t < 0 || t >= T) return;                       // out of range: nothing is written
  const size_t dst = (static_cast<size_t>(row) * T + t) * 64 + lane16 * 4;
  const float4 k = __ldg(reinterpret_cast<const float4*>(Knew + row * 64) + lane16);
  const float4 v = __ldg(reinterpret_cast<const float4*>(Vnew + row * 64) + lane16);
  if (cache_bf16) {
    __nv_bfloat162 k01 = __floats2bfloat162_rn(k.x, k.y), k23 = __floats2bfloat162_rn(k.z, k.w);
    __nv_bfloat162 v01 = __floats2bfloat162_rn(v.x, v.y), v23 = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(Kc) + dst) =
        make_uint2(*reinterpret_cast<uint32_t*>(&k01), *reinterpret_cast<uint32_t*>(&k23));
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(Vc) + dst) =
        make_uint2(*reinterpret_cast<uint32_t*>(&v01), *reinterpret_cast<uint32_t*>(&v23));
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(Kc) + dst) = k;
    *reinterpret_cast<float4*>(static_cast<float*>(Vc) + dst) = v;
  }
}

}  // namespace

cudaError_t launch_append(const AppendLaunch& a, cudaStream_t stream) {
  // No programmatic-launch trigger here: a decode that follows must not start
  // reading the cache before these rows are written.
  const long long rows = static_cast<long long>(a.B) * a.L * a.H;
  const long long grid = (rows + kAppendThreads / 16 - 1) / (kAppendThreads / 16);
  append_rows_kernel<<<static_cast<unsigned int>(grid), kAppendThreads, 0, stream>>>(
      a.pos, a.K_new, a.V_new, a.Kc, a.Vc, a.B, a.L * a.H, a.T, a.cache_bf16 ? 1 : 0);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace cxa
