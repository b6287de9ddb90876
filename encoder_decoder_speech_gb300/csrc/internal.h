// Internal interface between the C-ABI layer (cxa_api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <string>

#include <cuda_runtime.h>

struct cxa_cache;   // the C ABI's opaque descriptor (cxa_api.cu)

namespace cxa {

// Everything a populate launch needs; pointers are device pointers already
// validated by the C-ABI layer.
struct PopulateLaunch {
  void* Kc;            // cache bases (slot 0)
  void* Vc;
  const void* E;       // [nb][T][d]
  const void* WK;      // [L][d][d] (d_in, d_out)
  const void* WV;
  const float* bV;     // [L][d]
  const void* wpack;   // [2*L*d][d] K-major packed weights (launch_pack_weights)
  int b0, nb, T, d, L, H;
  int B;               // slots of the cache (for the cache tensor maps)
  bool in_bf16;
  bool cache_bf16;
};

struct DecodeLaunch {
  const void* Kc;
  const void* Vc;
  const float* Q;      // [B][nq][L][H][64]
  const int* key_len;  // [B]
  float* out;          // [B][nq][L][H][64]
  int nq;              // query rows per cache row (1..8)
  int l0, nl;          // decoded layers [l0, l0 + nl) of the cache's L
  int key_len_add;     // valid keys = clamp(key_len[b] + key_len_add, 0, T)
  void* workspace;
  int B, T, L, H;
  float scale;         // > 0
  bool cache_bf16;
  const float* K_new = nullptr;   // self-attention step: rows appended at key_len[b] (nq == 1)
  const float* V_new = nullptr;
};

// One decoder layer's cross-attention block for one step (see block.cu).
struct BlockLaunch {
  const void* Kc;
  const void* Vc;
  float* x;              // [B][d] residual stream, updated in place
  const float* gamma;    // [d] or NULL (1)
  const float* beta;     // [d] or NULL (0)
  float eps;
  const float* WQ;       // [d][d] (d_in, d_out)
  const float* bQ;       // [d] or NULL
  const float* WO;       // [d][d]
  const float* bO;       // [d] or NULL
  const int* key_len;    // [B]
  void* workspace;
  int B, T, L, H, layer;
  float scale;
  bool cache_bf16;
};

// One new K/V row per (slot, layer, head) written at position pos[b] (append.cu).
struct AppendLaunch {
  void* Kc;
  void* Vc;
  const int* pos;        // [B] device
  const float* K_new;    // [B][L][H][64]
  const float* V_new;
  int B, T, L, H;
  bool cache_bf16;
};

// Selected (layer, head) pairs, passed by value as a kernel parameter.
constexpr int kMaxAlignHeads = 64;
struct AlignHeads {
  int n;
  int l[kMaxAlignHeads];
  int h[kMaxAlignHeads];
};

// Cross-attention weights of selected heads (alignment.cu).
struct AlignLaunch {
  const void* Kc;
  const float* Q;        // [B][L][H][64]
  const int* key_len;    // [B]
  float* weights;        // [B][nsel][T]
  float* mean;           // [B][T] or NULL
  AlignHeads heads;
  int B, T, L, H;
  float scale;
  bool cache_bf16;
};

// Device facts of the current device, queried once per device.
struct DeviceInfo {
  int device;
  int num_sms;
  int cc_major, cc_minor;
  unsigned int* status_word;   // device address of the library's status word
};

// Fills *info for the current device; returns a CUDA error and a message on failure.
cudaError_t current_device_info(DeviceInfo* info, std::string* msg);

// Workspace layout helpers shared by the size query and the launchers.
size_t populate_workspace_bytes(int d, int L, bool in_bf16);
size_t decode_workspace_bytes(int B, int T, int L, int H, int nq);

// Launchers: enqueue on `stream`, return cudaSuccess or the first error; on a
// non-CUDA failure (e.g. tensor-map encoding) they return cudaErrorInvalidValue
// and describe it in *msg.
cudaError_t launch_populate(const PopulateLaunch& a, const DeviceInfo& dev, cudaStream_t stream,
                            std::string* msg);
// WK/WV [L][d][d] (d_in, d_out) -> the K-major operand layout of the populate GEMM
// (fp32 weights rounded to TF32), into wpack of populate_workspace_bytes(d, L, in_bf16).
cudaError_t launch_pack_weights(const void* WK, const void* WV, void* wpack, int d, int L, bool in_bf16,
                                cudaStream_t stream);
// n fp32 values -> bf16 (round to nearest even); src and dst 16-byte aligned.
cudaError_t launch_convert_bf16(const float* src, void* dst, size_t n, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_decode(const DecodeLaunch& a, const DeviceInfo& dev, cudaStream_t stream,
                          std::string* msg);
cudaError_t launch_block(const BlockLaunch& a, const DeviceInfo& dev, cudaStream_t stream, std::string* msg);
cudaError_t launch_append(const AppendLaunch& a, cudaStream_t stream);
// The latency shape of the one-query decode (decode_rows.cu): a cluster of CTAs per
// row. decode_rows_eligible says whether the policy lets `rows` rows of at most T
// keys take it; launch_decode_rows then launches it and sets *done, or leaves
// *done false (enqueuing nothing) when the rows' clusters cannot all be resident.
bool decode_rows_eligible(int rows, int T, int num_sms, int policy);
cudaError_t launch_decode_rows(const DecodeLaunch& a, const DeviceInfo& dev, cudaStream_t stream, bool* done);
cudaError_t launch_decode_shared_tc(const DecodeLaunch& a, const DeviceInfo& dev, cudaStream_t stream,
                                    std::string* msg);
cudaError_t launch_alignment(const AlignLaunch& a, const DeviceInfo& dev, cudaStream_t stream);
// The block as one kernel per layer: a cluster of H CTAs per slot (block_fused.cu).
bool fused_block_supported(int H, int dh);
// With *gathered set the launch did the whole block; otherwise it wrote the attention
// rows to att [B][d] and the out projection remains to be launched.
cudaError_t launch_block_fused(const BlockLaunch& a, float* att, bool* gathered, const DeviceInfo& dev,
                               cudaStream_t stream);
size_t block_workspace_bytes(int B, int T, int H);

// Bytes at the start of a decode workspace that hold the per-row arrival
// counters (the part that must be zero before a decode kernel starts).
size_t decode_counter_bytes(int B, int L, int H);

// Geometry of a cache descriptor (false for a NULL descriptor).
bool cache_geometry(const cxa_cache* c, int* B, int* T, int* L, int* H, int* dh);

// Number of times cxa_device_status has found the status word set (a kernel's
// bounded wait expired) in this process; scratch that a timed-out kernel may have
// left dirty is cleared again when this number changes.
unsigned long long timeout_epoch();

// The process-wide decode shape policy (cxa_set_decode_policy).
int decode_policy();
// The process-wide populate shape policy (cxa_set_populate_policy).
int populate_policy();

// Records the calling thread's last failure text (cxa_last_error_message).
void set_last_error(const std::string& msg);

// Counts every kernel launch the library makes.
void count_launches(unsigned long long n);

}  // namespace cxa
