// cxa_decode_noalloc: the decode step for callers that cannot allocate device
// memory (a host whose device memory all belongs to its own pool allocator, or
// a serving loop that must not pay for a fresh cudaMalloc). The source pages
// have no counterpart; this is an addition of the library.
//
// The scratch that cxa_decode takes from its caller (split-T partials and the
// per-row arrival counters) lives here in a file-scope device array instead.
// It is part of libcxa's device module, so every GPU that loads the library
// holds CXA_NOALLOC_SCRATCH_BYTES of it until the process exits. This entry
// point calls no cudaMalloc, cudaFree or other allocating routine.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>

#include "cxa.h"
#include "internal.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[CXA_NOALLOC_SCRATCH_BYTES];

namespace {

int noalloc_fail(int code, const std::string& msg) {
  cxa::set_last_error(msg);
  return code;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current.
cudaError_t scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[128] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int cxa_decode_noalloc(const cxa_cache* c, const float* Q, const int* key_len, float* out,
                                  float scale, void* stream) {
  int B, T, L, H, dh;
  if (!cxa::cache_geometry(c, &B, &T, &L, &H, &dh))
    return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: cache descriptor is NULL");
  const size_t need = cxa_decode_workspace_bytes(B, T, L, H, dh);
  if (need == 0 || need > CXA_NOALLOC_SCRATCH_BYTES)
    return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: this cache needs " + std::to_string(need) +
                                        " bytes of decode scratch, more than the fixed maximum of " +
                                        std::to_string(CXA_NOALLOC_SCRATCH_BYTES) +
                                        " bytes; use cxa_decode with a caller-owned workspace");
  // The checks cxa_decode makes, repeated here so that nothing (not even the
  // counter clear below) is enqueued for a call that is going to fail.
  if (Q == nullptr || key_len == nullptr || out == nullptr)
    return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: a pointer argument is NULL");
  if (!is_aligned(Q, 16) || !is_aligned(out, 16) || !is_aligned(key_len, 4))
    return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: Q and out must be 16-byte aligned");
  if (static_cast<const void*>(Q) == static_cast<const void*>(out))
    return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: out must not alias Q");
  if (!std::isfinite(scale)) return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: scale must be finite");
  for (int b = 0; b < B; ++b)
    if (cxa_is_ready(c, b) != 1)
      return noalloc_fail(CXA_ENOTREADY, "cxa_decode_noalloc: slot " + std::to_string(b) + " is not populated");

  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return noalloc_fail(CXA_ECUDA, std::string("cxa_decode_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));

  // The array keeps whatever the previous call left in it: start the arrival
  // counters of this geometry from zero.
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(scratch, 0, cxa::decode_counter_bytes(B, L, H), s);
  if (e != cudaSuccess)
    return noalloc_fail(CXA_ECUDA, std::string("cxa_decode_noalloc: clearing counters: ") + cudaGetErrorString(e));
  return cxa_decode(c, Q, key_len, out, scale, scratch, CXA_NOALLOC_SCRATCH_BYTES, stream);
}
