// The C ABI of libcxa (declared in include/cxa.h): the cache descriptor with its
// per-slot ready flags, argument validation, and dispatch to the kernel files.
// Every check runs before any device work is enqueued.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "cxa.h"
#include "internal.h"
#include "ptx.cuh"

// Device-side status word: kernels OR in 1 when a bounded wait expires.
static __device__ unsigned int g_cxa_status_word = 0;

struct cxa_cache {
  void* Kc;
  void* Vc;
  int B, T, L, H, dh;
  int dtype;
  std::vector<uint8_t> ready;   // populate sets, invalidate clears ("encoder_kv_ready")
  // What filled the cache, fixed by the first successful writer: projections of
  // encoder memory (cxa_populate) or self-attention rows (cxa_cache_append /
  // cxa_self_attention_step). The other kind of writer is refused, so an append
  // can never mark a stale (invalidated) cross-attention slot ready again.
  int role;
};

namespace {
constexpr int kRoleNone = 0, kRoleCross = 1, kRoleSelf = 2;
}

namespace {

thread_local std::string g_last_msg;
std::atomic<unsigned long long> g_launches{0};
std::atomic<unsigned long long> g_timeouts_seen{0};
std::atomic<int> g_decode_policy{CXA_DECODE_AUTO};
std::atomic<int> g_populate_policy{CXA_POPULATE_AUTO};

int fail(int code, const std::string& msg) {
  g_last_msg = msg;
  return code;
}

int fail_cuda(cudaError_t e, const std::string& what) {
  g_last_msg = what + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return CXA_ECUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_dtype(int t) { return t == CXA_F32 || t == CXA_BF16; }

}  // namespace

namespace cxa {

void count_launches(unsigned long long n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

cudaError_t current_device_info(DeviceInfo* info, std::string* msg) {
  static std::mutex mu;
  static DeviceInfo cache[128];
  static bool have[128] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *msg = "cudaGetDevice";
    return e;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 128 && have[dev]) {
    *info = cache[dev];
    return cudaSuccess;
  }
  DeviceInfo d{};
  d.device = dev;
  if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) {
    *msg = "cudaDeviceGetAttribute";
    return e;
  }
  if (d.cc_major != 10 || d.cc_minor != 3) {
    *msg = "libcxa is built for sm_103a (GB300); device " + std::to_string(dev) + " is sm_" +
           std::to_string(d.cc_major) + std::to_string(d.cc_minor);
    return cudaErrorNoKernelImageForDevice;
  }
  void* sym = nullptr;
  if ((e = cudaGetSymbolAddress(&sym, g_cxa_status_word)) != cudaSuccess) {
    *msg = "cudaGetSymbolAddress(status word)";
    return e;
  }
  d.status_word = static_cast<unsigned int*>(sym);
  if (dev >= 0 && dev < 128) {
    cache[dev] = d;
    have[dev] = true;
  }
  *info = d;
  return cudaSuccess;
}

void set_last_error(const std::string& msg) { g_last_msg = msg; }

unsigned long long timeout_epoch() { return g_timeouts_seen.load(std::memory_order_acquire); }

int decode_policy() { return g_decode_policy.load(std::memory_order_relaxed); }
int populate_policy() { return g_populate_policy.load(std::memory_order_relaxed); }

bool cache_geometry(const cxa_cache* c, int* B, int* T, int* L, int* H, int* dh) {
  if (c == nullptr) return false;
  *B = c->B;
  *T = c->T;
  *L = c->L;
  *H = c->H;
  *dh = c->dh;
  return true;
}

}  // namespace cxa

namespace cxa {
namespace {

// Failure-detection self-test: one thread waits, through the same bounded wait the
// kernels use, on an mbarrier that nothing ever arrives on; when the limit expires it
// sets the device status word, as a kernel whose copies never land would, and returns.
__global__ void wait_timeout_selftest_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    if (!mbar_wait(smem_u32(&bar), 0u, nullptr, limit_ns)) atomicOr(status, 1u);
  }
}

}  // namespace
}  // namespace cxa

extern "C" {

int cxa_cache_create(cxa_cache** out, void* Kc, void* Vc, int B, int T, int L, int H, int dh,
                     int cache_dtype) {
  if (out == nullptr) return fail(CXA_EINVAL, "cxa_cache_create: out is NULL");
  *out = nullptr;
  if (Kc == nullptr || Vc == nullptr) return fail(CXA_EINVAL, "cxa_cache_create: Kc or Vc is NULL");
  if (!aligned(Kc, 16) || !aligned(Vc, 16))
    return fail(CXA_EINVAL, "cxa_cache_create: Kc and Vc must be 16-byte aligned");
  if (T <= 0) return fail(CXA_EINVAL, "cxa_cache_create: the encoder memory length T must be positive");
  if (B <= 0 || L <= 0 || H <= 0) return fail(CXA_EINVAL, "cxa_cache_create: B, L and H must be positive");
  if (dh != 64) return fail(CXA_EINVAL, "cxa_cache_create: this build supports head_dim 64 only");
  if (!valid_dtype(cache_dtype)) return fail(CXA_EINVAL, "cxa_cache_create: cache_dtype must be CXA_F32 or CXA_BF16");
  if (static_cast<long long>(B) * L * H > 65535LL * 65535LL)
    return fail(CXA_EINVAL, "cxa_cache_create: too many (slot, layer, head) rows");
  if (L * H > 65535 || B > 65535) return fail(CXA_EINVAL, "cxa_cache_create: L*H and B must be <= 65535");
  cxa_cache* c = new (std::nothrow) cxa_cache;
  if (c == nullptr) return fail(CXA_EINVAL, "cxa_cache_create: out of host memory");
  c->Kc = Kc;
  c->Vc = Vc;
  c->B = B;
  c->T = T;
  c->L = L;
  c->H = H;
  c->dh = dh;
  c->dtype = cache_dtype;
  c->ready.assign(static_cast<size_t>(B), 0);
  c->role = kRoleNone;
  *out = c;
  return CXA_OK;
}

void cxa_cache_destroy(cxa_cache* c) { delete c; }

size_t cxa_populate_workspace_bytes(int d, int L, int in_dtype) {
  if (d <= 0 || L <= 0 || !valid_dtype(in_dtype)) return 0;
  return cxa::populate_workspace_bytes(d, L, in_dtype == CXA_BF16);
}

size_t cxa_decode_workspace_bytes(int B, int T, int L, int H, int dh) {
  if (B <= 0 || T <= 0 || L <= 0 || H <= 0 || dh != 64) return 0;
  return cxa::decode_workspace_bytes(B, T, L, H, 1);
}

size_t cxa_decode_shared_workspace_bytes(int B, int T, int L, int H, int dh, int nq) {
  // (the fp32-cache limit of 8 queries is checked by cxa_decode_shared)
  if (B <= 0 || T <= 0 || L <= 0 || H <= 0 || dh != 64 || nq < 1 || nq > CXA_MAX_SHARED_QUERIES) return 0;
  return cxa::decode_workspace_bytes(B, T, L, H, nq);
}

// Checks shared by the populate entry points (everything but the weights).
static int populate_checks(const char* who, cxa_cache* c, int b0, int nb, const void* E, const float* bV, int T,
                           int d, int L, int H, int in_dtype) {
  const std::string w(who);
  if (c == nullptr) return fail(CXA_EINVAL, w + ": cache descriptor is NULL");
  if (T <= 0) return fail(CXA_EINVAL, w + ": the encoder memory length T must be positive");
  if (H <= 0 || H * c->dh != d) return fail(CXA_EINVAL, w + ": num_heads * head_dim must equal the model width d");
  if (T != c->T || L != c->L || H != c->H) return fail(CXA_EINVAL, w + ": T, L, H do not match the cache descriptor");
  if (nb <= 0 || b0 < 0 || b0 + nb > c->B) return fail(CXA_EINVAL, w + ": slots [b0, b0+nb) out of range");
  if (!valid_dtype(in_dtype)) return fail(CXA_EINVAL, w + ": in_dtype must be CXA_F32 or CXA_BF16");
  if (E == nullptr || bV == nullptr) return fail(CXA_EINVAL, w + ": a pointer argument is NULL");
  if (!aligned(E, 16) || !aligned(bV, 16)) return fail(CXA_EINVAL, w + ": E and bV must be 16-byte aligned");
  if (c->role == kRoleSelf)
    return fail(CXA_EINVAL, w + ": this cache holds self-attention rows (cxa_cache_append); populate a cache of "
                                "its own");
  return CXA_OK;
}

static int check_weights(const char* who, const void* WK, const void* WV, int in_dtype) {
  const std::string w(who);
  if (WK == nullptr || WV == nullptr) return fail(CXA_EINVAL, w + ": WK or WV is NULL");
  const int esz = in_dtype == CXA_BF16 ? 2 : 4;
  if (!aligned(WK, esz) || !aligned(WV, esz))
    return fail(CXA_EINVAL, w + ": WK and WV must be aligned to their element size");
  return CXA_OK;
}

static int check_packed(const char* who, const void* packed, size_t packed_bytes, int d, int L, int in_dtype) {
  const std::string w(who);
  if (packed == nullptr) return fail(CXA_EINVAL, w + ": the packed-weight buffer is NULL");
  if (!aligned(packed, 256)) return fail(CXA_EINVAL, w + ": the packed-weight buffer must be 256-byte aligned");
  if (packed_bytes < cxa::populate_workspace_bytes(d, L, in_dtype == CXA_BF16))
    return fail(CXA_EINVAL, w + ": packed-weight buffer smaller than cxa_populate_workspace_bytes()");
  return CXA_OK;
}

// Enqueue the populate GEMM from packed weights; the slots are not ready until it
// is enqueued (and stay not ready if anything fails).
static int populate_enqueue(const char* who, cxa_cache* c, int b0, int nb, const void* E, const void* WK,
                            const void* WV, const void* packed, const float* bV, int T, int d, int L, int H,
                            int in_dtype, void* stream) {
  const std::string w(who);
  // New encoder memory: these slots are stale until the kernels are enqueued.
  for (int b = b0; b < b0 + nb; ++b) c->ready[static_cast<size_t>(b)] = 0;

  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, w + ": " + msg);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (WK != nullptr) {   // pack into the caller's workspace first
    e = cxa::launch_pack_weights(WK, WV, const_cast<void*>(packed), d, L, in_dtype == CXA_BF16, s);
    if (e != cudaSuccess) return fail_cuda(e, w + ": weight packing launch");
  }
  cxa::PopulateLaunch a;
  a.Kc = c->Kc;
  a.Vc = c->Vc;
  a.E = E;
  a.WK = WK;
  a.WV = WV;
  a.bV = bV;
  a.wpack = packed;
  a.b0 = b0;
  a.nb = nb;
  a.B = c->B;
  a.T = T;
  a.d = d;
  a.L = L;
  a.H = H;
  a.in_bf16 = in_dtype == CXA_BF16;
  a.cache_bf16 = c->dtype == CXA_BF16;
  e = cxa::launch_populate(a, dev, s, &msg);
  if (e != cudaSuccess) {
    if (!msg.empty()) return fail(CXA_EINVAL, w + ": " + msg);
    return fail_cuda(e, w + ": launch");
  }
  for (int b = b0; b < b0 + nb; ++b) c->ready[static_cast<size_t>(b)] = 1;
  c->role = kRoleCross;
  return CXA_OK;
}

int cxa_populate(cxa_cache* c, int b0, int nb, const void* E, const void* WK, const void* WV,
                 const float* bV, int T, int d, int L, int H, int in_dtype, void* workspace,
                 size_t workspace_bytes, void* stream) {
  int rc = populate_checks("cxa_populate", c, b0, nb, E, bV, T, d, L, H, in_dtype);
  if (rc == CXA_OK) rc = check_weights("cxa_populate", WK, WV, in_dtype);
  if (rc == CXA_OK) rc = check_packed("cxa_populate", workspace, workspace_bytes, d, L, in_dtype);
  if (rc != CXA_OK) return rc;
  return populate_enqueue("cxa_populate", c, b0, nb, E, WK, WV, workspace, bV, T, d, L, H, in_dtype, stream);
}

int cxa_pack_weights(const void* WK, const void* WV, int d, int L, int in_dtype, void* packed, size_t packed_bytes,
                     void* stream) {
  if (d <= 0 || d % 64 != 0 || L <= 0)
    return fail(CXA_EINVAL, "cxa_pack_weights: d must be a positive multiple of 64 and L positive");
  if (!valid_dtype(in_dtype)) return fail(CXA_EINVAL, "cxa_pack_weights: in_dtype must be CXA_F32 or CXA_BF16");
  int rc = check_weights("cxa_pack_weights", WK, WV, in_dtype);
  if (rc == CXA_OK) rc = check_packed("cxa_pack_weights", packed, packed_bytes, d, L, in_dtype);
  if (rc != CXA_OK) return rc;
  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, "cxa_pack_weights: " + msg);
  e = cxa::launch_pack_weights(WK, WV, packed, d, L, in_dtype == CXA_BF16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cxa_pack_weights: launch");
  return CXA_OK;
}

int cxa_convert_bf16(const float* src, void* dst, size_t n, void* stream) {
  if (src == nullptr || dst == nullptr) return fail(CXA_EINVAL, "cxa_convert_bf16: a pointer argument is NULL");
  if (!aligned(src, 16) || !aligned(dst, 16))
    return fail(CXA_EINVAL, "cxa_convert_bf16: src and dst must be 16-byte aligned");
  if (n == 0) return CXA_OK;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  if (s0 < d0 + 2 * n && d0 < s0 + 4 * n) return fail(CXA_EINVAL, "cxa_convert_bf16: src and dst overlap");
  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, "cxa_convert_bf16: " + msg);
  e = cxa::launch_convert_bf16(src, dst, n, dev, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cxa_convert_bf16: launch");
  return CXA_OK;
}

int cxa_populate_packed(cxa_cache* c, int b0, int nb, const void* E, const void* packed, size_t packed_bytes,
                        const float* bV, int T, int d, int L, int H, int in_dtype, void* stream) {
  int rc = populate_checks("cxa_populate_packed", c, b0, nb, E, bV, T, d, L, H, in_dtype);
  if (rc == CXA_OK) rc = check_packed("cxa_populate_packed", packed, packed_bytes, d, L, in_dtype);
  if (rc != CXA_OK) return rc;
  return populate_enqueue("cxa_populate_packed", c, b0, nb, E, nullptr, nullptr, packed, bV, T, d, L, H, in_dtype,
                          stream);
}

static int decode_common(const char* who, const cxa_cache* c, int l0, int nl, int nq, const float* Q,
                         const int* key_len, float* out, float scale, void* workspace, size_t workspace_bytes,
                         void* stream, int key_len_add = 0, const float* K_new = nullptr,
                         const float* V_new = nullptr) {
  const std::string w(who);
  if (c == nullptr) return fail(CXA_EINVAL, w + ": cache descriptor is NULL");
  if (nl == -1) nl = c->L;
  if (l0 < 0 || nl < 1 || l0 + nl > c->L) return fail(CXA_EINVAL, w + ": layers [l0, l0+nl) out of range");
  if (nq < 1 || nq > CXA_MAX_SHARED_QUERIES)
    return fail(CXA_EINVAL, w + ": nq must be in [1, " + std::to_string(CXA_MAX_SHARED_QUERIES) + "]");
  if (nq > CXA_MAX_SHARED_QUERIES_F32 && c->dtype == CXA_F32)
    return fail(CXA_EINVAL, w + ": an fp32 cache takes at most " + std::to_string(CXA_MAX_SHARED_QUERIES_F32) +
                                " queries per row");
  if (Q == nullptr || key_len == nullptr || out == nullptr || workspace == nullptr)
    return fail(CXA_EINVAL, w + ": a pointer argument is NULL");
  if (!aligned(Q, 16) || !aligned(out, 16) || !aligned(key_len, 4) || !aligned(workspace, 256))
    return fail(CXA_EINVAL, w + ": Q and out must be 16-byte aligned, the workspace 256-byte aligned");
  if (static_cast<const void*>(Q) == static_cast<const void*>(out))
    return fail(CXA_EINVAL, w + ": out must not alias Q");
  if (!std::isfinite(scale)) return fail(CXA_EINVAL, w + ": scale must be finite");
  if (workspace_bytes < cxa::decode_workspace_bytes(c->B, c->T, nl, c->H, nq))
    return fail(CXA_EINVAL, w + ": workspace smaller than the decode workspace size query");
  for (int b = 0; b < c->B; ++b)
    if (!c->ready[static_cast<size_t>(b)])
      return fail(CXA_ENOTREADY, w + ": slot " + std::to_string(b) +
                                     " is not populated (invalidated or never populated)");

  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, w + ": " + msg);

  cxa::DecodeLaunch a;
  a.Kc = c->Kc;
  a.Vc = c->Vc;
  a.Q = Q;
  a.key_len = key_len;
  a.out = out;
  a.nq = nq;
  a.l0 = l0;
  a.nl = nl;
  a.key_len_add = key_len_add;
  a.workspace = workspace;
  a.B = c->B;
  a.T = c->T;
  a.L = c->L;
  a.H = c->H;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(c->dh));
  a.cache_bf16 = c->dtype == CXA_BF16;
  a.K_new = K_new;
  a.V_new = V_new;
  e = cxa::launch_decode(a, dev, static_cast<cudaStream_t>(stream), &msg);
  if (e != cudaSuccess) return fail_cuda(e, w + ": launch");
  return CXA_OK;
}

int cxa_decode(const cxa_cache* c, const float* Q, const int* key_len, float* out, float scale,
               void* workspace, size_t workspace_bytes, void* stream) {
  return decode_common("cxa_decode", c, 0, -1, 1, Q, key_len, out, scale, workspace, workspace_bytes, stream);
}

int cxa_decode_layers(const cxa_cache* c, int l0, int nl, const float* Q, const int* key_len, float* out,
                      float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (nl < 1) return fail(CXA_EINVAL, "cxa_decode_layers: nl must be >= 1");
  return decode_common("cxa_decode_layers", c, l0, nl, 1, Q, key_len, out, scale, workspace, workspace_bytes,
                       stream);
}

int cxa_decode_shared(const cxa_cache* c, int nq, const float* Q, const int* key_len, float* out,
                      float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_common("cxa_decode_shared", c, 0, -1, nq, Q, key_len, out, scale, workspace, workspace_bytes,
                       stream);
}

int cxa_cache_append(cxa_cache* c, const int* pos, const float* K_new, const float* V_new, void* stream) {
  if (c == nullptr) return fail(CXA_EINVAL, "cxa_cache_append: cache descriptor is NULL");
  if (pos == nullptr || K_new == nullptr || V_new == nullptr)
    return fail(CXA_EINVAL, "cxa_cache_append: a pointer argument is NULL");
  if (!aligned(pos, 4) || !aligned(K_new, 16) || !aligned(V_new, 16))
    return fail(CXA_EINVAL, "cxa_cache_append: K_new and V_new must be 16-byte aligned");
  if (c->role == kRoleCross)
    return fail(CXA_EINVAL, "cxa_cache_append: this cache holds projections of encoder memory (cxa_populate); "
                            "appending would mark its invalidated slots ready");
  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, "cxa_cache_append: " + msg);
  cxa::AppendLaunch a;
  a.Kc = c->Kc;
  a.Vc = c->Vc;
  a.pos = pos;
  a.K_new = K_new;
  a.V_new = V_new;
  a.B = c->B;
  a.T = c->T;
  a.L = c->L;
  a.H = c->H;
  a.cache_bf16 = c->dtype == CXA_BF16;
  e = cxa::launch_append(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cxa_cache_append: launch");
  for (auto& r : c->ready) r = 1;
  c->role = kRoleSelf;
  return CXA_OK;
}

int cxa_self_attention_step(cxa_cache* c, const int* pos, const float* Q, const float* K_new, const float* V_new,
                            float* out, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (c == nullptr) return fail(CXA_EINVAL, "cxa_self_attention_step: cache descriptor is NULL");
  // every check of the decode first, so a failing call enqueues nothing
  if (Q == nullptr || out == nullptr || workspace == nullptr || pos == nullptr)
    return fail(CXA_EINVAL, "cxa_self_attention_step: a pointer argument is NULL");
  if (!aligned(Q, 16) || !aligned(out, 16) || !aligned(workspace, 256))
    return fail(CXA_EINVAL, "cxa_self_attention_step: Q and out must be 16-byte aligned, the workspace 256-byte aligned");
  if (static_cast<const void*>(Q) == static_cast<const void*>(out))
    return fail(CXA_EINVAL, "cxa_self_attention_step: out must not alias Q");
  if (!std::isfinite(scale)) return fail(CXA_EINVAL, "cxa_self_attention_step: scale must be finite");
  if (workspace_bytes < cxa::decode_workspace_bytes(c->B, c->T, c->L, c->H, 1))
    return fail(CXA_EINVAL, "cxa_self_attention_step: workspace smaller than cxa_decode_workspace_bytes()");
  if (K_new == nullptr || V_new == nullptr)
    return fail(CXA_EINVAL, "cxa_self_attention_step: a pointer argument is NULL");
  if (!aligned(pos, 4) || !aligned(K_new, 16) || !aligned(V_new, 16))
    return fail(CXA_EINVAL, "cxa_self_attention_step: K_new and V_new must be 16-byte aligned");
  if (c->role == kRoleCross)
    return fail(CXA_EINVAL, "cxa_self_attention_step: this cache holds projections of encoder memory "
                            "(cxa_populate); appending would mark its invalidated slots ready");
  // appending makes every slot a valid (partly filled) self-attention cache; the
  // flags are restored if the step fails before anything is enqueued
  std::vector<uint8_t> was = c->ready;
  for (auto& r : c->ready) r = 1;
  // one kernel: the append is fused into the decode over positions 0 .. pos[b]
  const int rc = decode_common("cxa_self_attention_step", c, 0, -1, 1, Q, pos, out, scale, workspace,
                               workspace_bytes, stream, 1, K_new, V_new);
  if (rc == CXA_OK) c->role = kRoleSelf;
  else c->ready.swap(was);
  return rc;
}

int cxa_alignment_weights(const cxa_cache* c, const float* Q, const int* key_len, const int* heads_lh, int nsel,
                          float* weights, float* mean, float scale, void* stream) {
  if (c == nullptr) return fail(CXA_EINVAL, "cxa_alignment_weights: cache descriptor is NULL");
  if (nsel < 1 || nsel > cxa::kMaxAlignHeads)
    return fail(CXA_EINVAL, "cxa_alignment_weights: nsel must be in [1, " + std::to_string(cxa::kMaxAlignHeads) + "]");
  if (Q == nullptr || key_len == nullptr || heads_lh == nullptr || weights == nullptr)
    return fail(CXA_EINVAL, "cxa_alignment_weights: a pointer argument is NULL");
  if (!aligned(Q, 16) || !aligned(key_len, 4) || !aligned(weights, 4) || (mean != nullptr && !aligned(mean, 4)))
    return fail(CXA_EINVAL, "cxa_alignment_weights: Q must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(CXA_EINVAL, "cxa_alignment_weights: scale must be finite");
  cxa::AlignHeads hs;
  hs.n = nsel;
  for (int k = 0; k < nsel; ++k) {
    const int l = heads_lh[2 * k], h = heads_lh[2 * k + 1];
    if (l < 0 || l >= c->L || h < 0 || h >= c->H)
      return fail(CXA_EINVAL, "cxa_alignment_weights: head " + std::to_string(k) + " out of range");
    hs.l[k] = l;
    hs.h[k] = h;
  }
  for (int b = 0; b < c->B; ++b)
    if (!c->ready[static_cast<size_t>(b)])
      return fail(CXA_ENOTREADY, "cxa_alignment_weights: slot " + std::to_string(b) + " is not populated");
  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, "cxa_alignment_weights: " + msg);
  cxa::AlignLaunch a;
  a.Kc = c->Kc;
  a.Q = Q;
  a.key_len = key_len;
  a.weights = weights;
  a.mean = mean;
  a.heads = hs;
  a.B = c->B;
  a.T = c->T;
  a.L = c->L;
  a.H = c->H;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(c->dh));
  a.cache_bf16 = c->dtype == CXA_BF16;
  e = cxa::launch_alignment(a, dev, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cxa_alignment_weights: launch");
  return CXA_OK;
}

size_t cxa_cross_block_workspace_bytes(int B, int T, int L, int H, int dh) {
  if (B <= 0 || T <= 0 || L <= 0 || H <= 0 || dh != 64) return 0;
  return cxa::block_workspace_bytes(B, T, H);
}

int cxa_cross_block(const cxa_cache* c, int layer, float* x, const float* ln_gamma, const float* ln_beta,
                    float ln_eps, const float* WQ, const float* bQ, const float* WO, const float* bO,
                    const int* key_len, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (c == nullptr) return fail(CXA_EINVAL, "cxa_cross_block: cache descriptor is NULL");
  if (layer < 0 || layer >= c->L) return fail(CXA_EINVAL, "cxa_cross_block: layer out of range");
  if (x == nullptr || WQ == nullptr || WO == nullptr || key_len == nullptr || workspace == nullptr)
    return fail(CXA_EINVAL, "cxa_cross_block: a required pointer argument is NULL");
  if (!aligned(x, 16) || !aligned(WQ, 16) || !aligned(WO, 16) || !aligned(workspace, 256) || !aligned(key_len, 4))
    return fail(CXA_EINVAL, "cxa_cross_block: x, WQ and WO must be 16-byte aligned, the workspace 256-byte aligned");
  if (!std::isfinite(scale) || !std::isfinite(ln_eps) || ln_eps < 0.f)
    return fail(CXA_EINVAL, "cxa_cross_block: scale and ln_eps must be finite, ln_eps >= 0");
  if (workspace_bytes < cxa::block_workspace_bytes(c->B, c->T, c->H))
    return fail(CXA_EINVAL, "cxa_cross_block: workspace smaller than cxa_cross_block_workspace_bytes()");
  for (int b = 0; b < c->B; ++b)
    if (!c->ready[static_cast<size_t>(b)])
      return fail(CXA_ENOTREADY, "cxa_cross_block: slot " + std::to_string(b) + " is not populated");
  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, "cxa_cross_block: " + msg);
  cxa::BlockLaunch a;
  a.Kc = c->Kc;
  a.Vc = c->Vc;
  a.x = x;
  a.gamma = ln_gamma;
  a.beta = ln_beta;
  a.eps = ln_eps;
  a.WQ = WQ;
  a.bQ = bQ;
  a.WO = WO;
  a.bO = bO;
  a.key_len = key_len;
  a.workspace = workspace;
  a.B = c->B;
  a.T = c->T;
  a.L = c->L;
  a.H = c->H;
  a.layer = layer;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(c->dh));
  a.cache_bf16 = c->dtype == CXA_BF16;
  e = cxa::launch_block(a, dev, static_cast<cudaStream_t>(stream), &msg);
  if (e != cudaSuccess) {
    if (!msg.empty()) return fail(CXA_EINVAL, "cxa_cross_block: " + msg);
    return fail_cuda(e, "cxa_cross_block: launch");
  }
  return CXA_OK;
}

int cxa_invalidate(cxa_cache* c, int b) {
  if (c == nullptr) return fail(CXA_EINVAL, "cxa_invalidate: cache descriptor is NULL");
  if (b == -1) {
    for (auto& r : c->ready) r = 0;
    return CXA_OK;
  }
  if (b < 0 || b >= c->B) return fail(CXA_EINVAL, "cxa_invalidate: slot out of range");
  c->ready[static_cast<size_t>(b)] = 0;
  return CXA_OK;
}

int cxa_is_ready(const cxa_cache* c, int b) {
  if (c == nullptr || b < 0 || b >= c->B) return CXA_EINVAL;
  return c->ready[static_cast<size_t>(b)] ? 1 : 0;
}

const char* cxa_strerror(int code) {
  switch (code) {
    case CXA_OK: return "CXA_OK";
    case CXA_EINVAL: return "CXA_EINVAL: invalid argument or geometry";
    case CXA_ENOTREADY: return "CXA_ENOTREADY: projection cache not populated";
    case CXA_ECUDA: return "CXA_ECUDA: CUDA runtime error";
    case CXA_ETIMEOUT: return "CXA_ETIMEOUT: a kernel's bounded wait expired";
    default: return "unknown cxa status";
  }
}

const char* cxa_last_error_message(void) { return g_last_msg.c_str(); }

unsigned long long cxa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int cxa_set_decode_policy(int policy) {
  if (policy != CXA_DECODE_AUTO && policy != CXA_DECODE_STREAM && policy != CXA_DECODE_ROWS)
    return fail(CXA_EINVAL, "cxa_set_decode_policy: unknown policy");
  g_decode_policy.store(policy, std::memory_order_relaxed);
  return CXA_OK;
}

int cxa_set_populate_policy(int policy) {
  if (policy != CXA_POPULATE_AUTO && policy != CXA_POPULATE_PAIR && policy != CXA_POPULATE_SINGLE)
    return fail(CXA_EINVAL, "cxa_set_populate_policy: unknown policy");
  g_populate_policy.store(policy, std::memory_order_relaxed);
  return CXA_OK;
}

int cxa_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000)
    return fail(CXA_EINVAL, "cxa_selftest_wait_timeout: limit_us must be in [1, 1000000]");
  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, "cxa_selftest_wait_timeout: " + msg);
  cxa::wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      dev.status_word, static_cast<unsigned long long>(limit_us) * 1000ull);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail_cuda(e, "cxa_selftest_wait_timeout: launch");
  cxa::count_launches(1);
  return CXA_OK;
}

int cxa_device_status(int clear) {
  std::string msg;
  cxa::DeviceInfo dev;
  cudaError_t e = cxa::current_device_info(&dev, &msg);
  if (e != cudaSuccess) return fail_cuda(e, "cxa_device_status: " + msg);
  unsigned int word = 0;
  if ((e = cudaMemcpy(&word, dev.status_word, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail_cuda(e, "cxa_device_status: read");
  if (word) g_timeouts_seen.fetch_add(1, std::memory_order_acq_rel);
  if (clear) {
    const unsigned int zero = 0;
    if ((e = cudaMemcpy(dev.status_word, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
      return fail_cuda(e, "cxa_device_status: clear");
  }
  return word ? CXA_ETIMEOUT : CXA_OK;
}

}  // extern "C"
