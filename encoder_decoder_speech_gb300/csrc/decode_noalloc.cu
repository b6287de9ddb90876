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
//
// What must start at zero is the arrival counters. The decode kernel leaves
// every counter it touches at zero when it completes (the last arriver of a
// split row resets it; whole rows never touch theirs), whatever the geometry of
// the call, and it writes every partial before any CTA reads it. So the array
// is cleared only when this file sets it up in a CUDA context and again after
// cxa_device_status has reported a timed-out kernel (which may have stopped
// between a counter increment and its reset) -- not on every call, so that a
// call overlaps the kernel before it through programmatic dependent launch as
// cxa_decode does.
#include <cuda.h>
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

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent from the driver, through the runtime's entry-point query (no
// link against libcuda); nullptr if the driver does not offer it.
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  return fn;
}

// Device address of g_noalloc_scratch in the current CUDA context. In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress, with the device current: once per device and
// context (a device reset or a new context reloads the module, and the array may
// then sit elsewhere; without the driver's context query it is looked up on
// every call). *clear is set when the array must be zeroed before this call: on
// set-up, and when cxa_device_status has seen a timeout since the last clear.
cudaError_t scratch_address(void** out, bool* clear) {
  struct State {
    void* addr = nullptr;
    CUcontext ctx = nullptr;
    unsigned long long epoch = 0;
  };
  static std::mutex mu;
  static State state[128];
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  CUcontext ctx = nullptr;
  const CtxGetCurrentFn get = ctx_get_current();
  const bool have_ctx = get != nullptr && get(&ctx) == CUDA_SUCCESS && ctx != nullptr;
  const unsigned long long epoch = cxa::timeout_epoch();
  std::lock_guard<std::mutex> lock(mu);
  State& st = state[dev];
  *clear = false;
  if (st.addr == nullptr || !have_ctx || ctx != st.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (st.addr == nullptr || (have_ctx && ctx != st.ctx)) *clear = true;
    st.addr = p;
    st.ctx = have_ctx ? ctx : nullptr;
    st.epoch = epoch;
  }
  if (st.epoch != epoch) {
    *clear = true;
    st.epoch = epoch;
  }
  *out = st.addr;
  return cudaSuccess;
}

}  // namespace

extern "C" int cxa_decode_noalloc(const cxa_cache* c, const float* Q, const int* key_len, float* out,
                                  float scale, void* stream) {
  int B, T, L, H, dh;
  if (!cxa::cache_geometry(c, &B, &T, &L, &H, &dh))
    return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: cache descriptor is NULL");
  const size_t need = cxa_decode_workspace_bytes(B, T, L, H, dh);
  if (need == 0)
    return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: unsupported cache geometry (head_dim must be 64)");
  if (need > CXA_NOALLOC_SCRATCH_BYTES)
    return noalloc_fail(CXA_EINVAL, "cxa_decode_noalloc: this cache needs " + std::to_string(need) +
                                        " bytes of decode scratch, more than the fixed maximum of " +
                                        std::to_string(CXA_NOALLOC_SCRATCH_BYTES) +
                                        " bytes; use cxa_decode with a caller-owned workspace");
  // The checks cxa_decode makes, repeated here so that nothing (not even a
  // scratch clear) is enqueued for a call that is going to fail.
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
  bool clear = false;
  cudaError_t e = scratch_address(&scratch, &clear);
  if (e != cudaSuccess)
    return noalloc_fail(CXA_ECUDA, std::string("cxa_decode_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (clear) {
    e = cudaMemsetAsync(scratch, 0, CXA_NOALLOC_SCRATCH_BYTES, s);
    if (e != cudaSuccess)
      return noalloc_fail(CXA_ECUDA, std::string("cxa_decode_noalloc: clearing the scratch: ") + cudaGetErrorString(e));
  }
  return cxa_decode(c, Q, key_len, out, scale, scratch, CXA_NOALLOC_SCRATCH_BYTES, stream);
}
