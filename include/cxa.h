/*
 * cxa.h -- C ABI of libcxa: encoder-decoder cross-attention on one GB300 (sm_103a).
 *
 * Two operations make up the path:
 *
 *   populate  K_l = E x WK_l and V_l = E x WV_l + bV_l for every decoder layer l,
 *             written straight into a layer-major, head-major K/V projection cache
 *             ("Whisper: Trace One Encoder Tensor into Every Decoder Layer",
 *             "The concept: one tensor, many consumers" for the formulas and the
 *             cache policy; "View 2 -- expand one cross-attention operation" for
 *             the per-layer slab; "Deliberate failure: token-major K meets a
 *             head-major consumer" for the token-major -> head-major re-layout).
 *   decode    one query row per (slot, layer, head) attends non-causally over all
 *             valid encoder keys: out = softmax(scale * q.K^T) V ("View 2": the
 *             decode call with num_heads, query_tokens = 1, key_tokens, head_dim
 *             and scale = 0.125 = 1/sqrt(64)).
 *
 * The cache is caller-owned explicit I/O ("Recurrence as feeds", "What it
 * opened": a cache is an extra input that one run writes and the next reads).
 * The library allocates no device memory: every device buffer below (E, weights,
 * biases, cache, queries, key lengths, outputs, workspaces) belongs to the caller
 * and must stay alive until the work enqueued on the stream has finished.
 * The descriptor (cxa_cache) is a small host object: geometry, dtype and the
 * per-slot ready flags.
 *
 * All calls that take a stream are asynchronous: they validate their arguments
 * on the host, enqueue kernels on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and return. Every check happens before any device work is enqueued,
 * so a call that returns an error has launched nothing.
 *
 * Status codes (int): CXA_OK on success, otherwise one of the negative codes
 * below; cxa_strerror() names a code and cxa_last_error_message() gives the
 * detail of the calling thread's last failure.
 */
#ifndef CXA_H_
#define CXA_H_

#include <stddef.h>

#if defined(__GNUC__)
#define CXA_API __attribute__((visibility("default")))
#else
#define CXA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define CXA_OK          0
#define CXA_EINVAL     (-1)  /* bad geometry, null or misaligned pointer, short workspace */
#define CXA_ENOTREADY  (-2)  /* a slot of the cache is not populated: decode refuses
                                ("View 3 -- prefill vs decode": decode refuses (-2)
                                until prefill repopulates the cache) */
#define CXA_ECUDA      (-3)  /* a CUDA runtime error (launch failure, wrong device) */
#define CXA_ETIMEOUT   (-4)  /* a kernel's bounded wait expired (see cxa_device_status) */

/* ---- element types ------------------------------------------------------- */
#define CXA_F32   0   /* IEEE fp32 */
#define CXA_BF16  1   /* bfloat16, stored as 16-bit words */

typedef struct cxa_cache cxa_cache;

/*
 * Create a cache descriptor over caller-owned K/V cache buffers.
 *
 *   Kc, Vc  device pointers, each B*L*H*T*dh elements of cache_dtype, laid out
 *           [B][L][H][T][dh] (slot, layer-major, head-major: element (b,l,h,t,c)
 *           at (((b*L + l)*H + h)*T + t)*dh + c; for one Whisper-Base slot in fp32
 *           the layer-5 K slab starts 15,360,000 bytes in, as "View 2" prints).
 *           16-byte aligned.
 *   B       batch slots (independent encoder memories), >= 1.
 *   T       encoder length T_enc, > 0 ("View 3": a positive encoder memory
 *           length is required).
 *   L, H    decoder layers and heads, >= 1.
 *   dh      head dimension; this build supports dh == 64 only.
 *   cache_dtype  CXA_F32 or CXA_BF16 (bf16 stores round to nearest even).
 *
 * Every slot starts not ready. Returns CXA_EINVAL on bad arguments (and leaves
 * *out NULL). Performs no CUDA call.
 */
CXA_API int cxa_cache_create(cxa_cache** out, void* Kc, void* Vc, int B, int T, int L, int H,
                     int dh, int cache_dtype);

/* Free the descriptor (not the caller's buffers). NULL is ignored. */
CXA_API void cxa_cache_destroy(cxa_cache* c);

/*
 * Bytes of the packed layer weights for width d, L layers and input type
 * in_dtype: WK and WV of every layer in the K-major operand layout of the
 * tensor-core GEMM (2*L*d*d elements of in_dtype). This is the size of
 * cxa_populate's workspace (which it packs into on every call) and of the buffer
 * cxa_pack_weights fills once for cxa_populate_packed.
 */
CXA_API size_t cxa_populate_workspace_bytes(int d, int L, int in_dtype);

/*
 * Bytes of device workspace cxa_decode needs for a cache of this geometry: one
 * partial softmax state (running max, running sum, dh accumulators) per
 * (slot, layer, head, key chunk), plus per-row arrival counters.
 */
CXA_API size_t cxa_decode_workspace_bytes(int B, int T, int L, int H, int dh);

/*
 * Populate slots [b0, b0+nb) of the cache from nb encoder memories.
 *
 *   E       device, [nb][T][d] of in_dtype, token-major (row t = one encoder
 *           frame), 16-byte aligned.
 *   WK, WV  device, [L][d][d] of in_dtype, each layer indexed (d_in, d_out) so
 *           that K_l = E x WK_l; head h owns output columns h*dh .. h*dh+dh-1.
 *   bV      device, [L][d] fp32 value bias, 16-byte aligned, added to V only. There is no key
 *           bias: it cannot change the softmax ("Caso de estudio: WhisperKit",
 *           §2: the key-projection bias is dropped as redundant).
 *   T, d, L, H   must match the descriptor, with H*dh == d ("View 3": num_heads *
 *           head_dim == embed_dim is a hard error).
 *   in_dtype CXA_F32 (tensor cores read the fp32 operands as TF32) or CXA_BF16.
 *   workspace, workspace_bytes  device scratch of at least
 *           cxa_populate_workspace_bytes(d, L, in_dtype) bytes, 256-byte aligned.
 *
 * The slots are marked not ready first and ready again once both kernels are
 * enqueued without error, so a failed call leaves them not ready. Readiness is
 * stream-ordered: decode on the same stream (or after an event) sees the data.
 * Refused with CXA_EINVAL on a cache that cxa_cache_append or
 * cxa_self_attention_step has written (a self-attention cache).
 *
 * Two kernels: the weight packing into `workspace`, then the GEMM. A caller that
 * populates many windows with the same weights packs them once instead
 * (cxa_pack_weights) and calls cxa_populate_packed.
 */
CXA_API int cxa_populate(cxa_cache* c, int b0, int nb, const void* E, const void* WK,
                 const void* WV, const float* bV, int T, int d, int L, int H,
                 int in_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Pack the layer weights once into the operand layout of the populate GEMM.
 * The decoder's WK_l / WV_l are static from one audio window to the next; only
 * the encoder memory E changes ("The concept: one tensor, many consumers": E is
 * projected once per layer at prefill, the weights belong to the model), so the
 * repack is done once, when the weights are loaded, not per window.
 *
 *   WK, WV   device, [L][d][d] of in_dtype, indexed (d_in, d_out) as for
 *            cxa_populate; d a positive multiple of 64.
 *   packed, packed_bytes  device buffer of at least
 *            cxa_populate_workspace_bytes(d, L, in_dtype) bytes, 256-byte aligned,
 *            owned by the caller; it keeps the packed weights until the caller
 *            overwrites it (fp32 weights are stored rounded to TF32, round to
 *            nearest, ties away from zero).
 * One kernel on `stream`. CXA_EINVAL for bad sizes or pointers.
 */
CXA_API int cxa_pack_weights(const void* WK, const void* WV, int d, int L, int in_dtype, void* packed,
                             size_t packed_bytes, void* stream);

/*
 * cxa_populate from weights packed by cxa_pack_weights (same d, L and in_dtype):
 * one kernel, the GEMM with its head-major epilogue. Arguments, ready-flag rules
 * and errors as for cxa_populate; `packed` must hold the packed weights when the
 * kernel runs (stream order).
 */
CXA_API int cxa_populate_packed(cxa_cache* c, int b0, int nb, const void* E, const void* packed,
                                size_t packed_bytes, const float* bV, int T, int d, int L, int H,
                                int in_dtype, void* stream);

/*
 * fp32 -> bf16 conversion, round to nearest even (NaN stays NaN, values beyond
 * the largest bf16 round to infinity): the pass in front of the bf16 populate
 * for an encoder memory that arrives in fp32 (the Whisper-large workload's
 * E [1500, 1280] fp32 populated with bf16 tensor-core inputs), or for fp32
 * weights before cxa_pack_weights with in_dtype CXA_BF16.
 *
 *   src   device fp32 [n], 16-byte aligned.
 *   dst   device bf16 [n] (16-bit words), 16-byte aligned; must not overlap src.
 * One kernel on `stream`; n == 0 enqueues nothing. CXA_EINVAL for NULL,
 * misaligned or overlapping buffers.
 */
CXA_API int cxa_convert_bf16(const float* src, void* dst, size_t n, void* stream);

/*
 * One decode step for every slot, layer and head.
 *
 *   Q        device fp32 [B][L][H][dh], one query row per (slot, layer, head);
 *            16-byte aligned.
 *   key_len  device int32 [B], valid encoder keys per slot; keys t >= key_len[b]
 *            are excluded exactly (the limit of the additive key-padding mask,
 *            "Caso de estudio: WhisperKit", §4). Values are clamped to [0, T];
 *            a slot with no valid key gets a zero output (the clamped softmax
 *            denominator of §2). Padded cache rows are never read.
 *   out      device fp32 [B][L][H][dh], 16-byte aligned; may not alias Q.
 *   scale    multiplies q.k; a value <= 0 selects 1/sqrt(dh).
 *   workspace, workspace_bytes  device scratch of at least
 *            cxa_decode_workspace_bytes(B, T, L, H, dh) bytes, 256-byte aligned;
 *            its counters must be zero before the first call on a new buffer
 *            (cudaMemset) and the kernels leave them zero afterwards. Calls that
 *            share a workspace must be ordered on one stream.
 *
 * Returns CXA_ENOTREADY, launching nothing, unless every slot is ready.
 *
 * Launch overlap: the decode kernel is launched with programmatic dependent
 * launch. When the kernel just before it on the stream allows that (the
 * library's own decode kernels do), the decode starts while that kernel drains
 * and reads the cache rows and key_len early; it waits for the earlier kernel
 * to finish before it reads Q or writes out or the workspace. So Q and out may
 * be produced and consumed by neighbouring kernels freely, but the cache and
 * key_len must not be written by an immediately preceding kernel that itself
 * triggers programmatic launch (an ordinary kernel, a copy or cxa_populate /
 * cxa_cache_append in between is always safe).
 */
CXA_API int cxa_decode(const cxa_cache* c, const float* Q, const int* key_len, float* out,
               float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Shared-cache decode: nq query rows per (slot, layer, head), all attending the
 * same cache slot -- the beam or speculative hypotheses of one audio window
 * share its encoder memory ("Caso de estudio: WhisperKit", §3: SharedSplitKVCached
 * attends one shared batch-1 cache from a batch-N query). Each K/V row is read
 * once per step for all nq queries.
 *
 *   nq       query rows per cache row, 1 .. CXA_MAX_SHARED_QUERIES (16) for a
 *            bf16 cache, 1 .. CXA_MAX_SHARED_QUERIES_F32 (8) for an fp32 cache.
 *            With a bf16 cache and nq >= 2 the scores run on the tensor cores
 *            (queries as bf16 hi + lo parts); otherwise in fp32 on the CUDA cores.
 *   Q, out   device fp32 [B][nq][L][H][dh]: row (b, n, l, h) is hypothesis n of
 *            slot b; out row (b, n, l, h) = softmax(scale * q.K[b,l,h]^T) V[b,l,h].
 *   key_len, scale  as for cxa_decode (key_len is per slot, shared by its rows).
 *   workspace, workspace_bytes  at least cxa_decode_shared_workspace_bytes(B, T,
 *            L, H, dh, nq) bytes, 256-byte aligned, with the same counter rules
 *            as cxa_decode's workspace.
 *
 * Launches: one kernel, or, with a bf16 cache and nq >= 5, two: the decode and a
 * small kernel that merges the rows whose keys were split between the decode's
 * CTAs (from the workspace's partial states, in segment order). Both use
 * programmatic dependent launch with the overlap rules of cxa_decode; the merge
 * kernel reads key_len early and everything else only after the decode grid has
 * finished, so the pair behaves like one decode towards the kernels around it.
 *
 * With nq = 1 this is exactly cxa_decode. Errors as for cxa_decode, and
 * CXA_EINVAL for nq outside those ranges.
 */
#define CXA_MAX_SHARED_QUERIES 16
#define CXA_MAX_SHARED_QUERIES_F32 8

CXA_API size_t cxa_decode_shared_workspace_bytes(int B, int T, int L, int H, int dh, int nq);

CXA_API int cxa_decode_shared(const cxa_cache* c, int nq, const float* Q, const int* key_len,
                              float* out, float scale, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Self-attention KV cache: append one row per (slot, layer, head) at position
 * pos[b] -- the new token's key and value of a decoder step ("Caso de estudio:
 * WhisperKit", §4: a fixed max_seq_len cache updated by a one-hot masked blend at
 * the current position; "Recurrence as feeds", "What it opened": the new rows
 * are written with scatter). A cache created with T = max_seq_len serves as the
 * decoder's self-attention cache: cxa_decode with key_len = pos + 1 then attends
 * positions 0 .. pos, the causal row of the whole-window formula.
 *
 *   pos      device int32 [B]; a slot whose pos is outside [0, T) is left as is.
 *   K_new, V_new  device fp32 [B][L][H][dh], 16-byte aligned (rounded to bf16
 *            for a bf16 cache).
 * Marks every slot ready (each slot is a partly filled self-attention cache).
 * Refused with CXA_EINVAL, launching nothing, on a cache that cxa_populate has
 * written: marking its slots ready would un-refuse an invalidated cross-attention
 * slot. Asynchronous on stream.
 */
CXA_API int cxa_cache_append(cxa_cache* c, const int* pos, const float* K_new, const float* V_new,
                             void* stream);

/*
 * One self-attention decoder step: cxa_cache_append(pos, K_new, V_new) then the
 * decode of Q over positions 0 .. pos[b] of every slot (key_len = pos + 1).
 * Arguments as for cxa_cache_append and cxa_decode (workspace of
 * cxa_decode_workspace_bytes size). Every argument is checked before anything
 * is enqueued; refused like cxa_cache_append on a populated cache.
 *
 * Launch overlap: one kernel, launched with programmatic dependent launch. It
 * streams slot b's cache rows t < min(pos[b], T) - 1 before the kernel just
 * before it on the stream has finished, and everything else (row pos[b] - 1,
 * which the previous step writes in a decoding loop, Q, the new rows, out) only
 * after. It lets the next kernel start only after that wait, so a step never
 * overlaps work older than its immediate predecessor. Hence the kernel just
 * before a step must not write rows t < pos[b] - 1 while launched with
 * programmatic launch: consecutive steps that advance pos[b] by at most one
 * (or move it back), and any cxa_cache_append, cxa_populate, ordinary kernel or
 * copy in between, are always safe.
 */
CXA_API int cxa_self_attention_step(cxa_cache* c, const int* pos, const float* Q, const float* K_new,
                                    const float* V_new, float* out, float scale, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Cross-attention weights of selected alignment heads for one decode step
 * ("Caso de estudio: WhisperKit", §6: the cross-attention of chosen alignment
 * heads returns its weights, and their mean over heads is returned as an extra
 * output for word timestamps):
 *
 *   weights[b][k][t] = softmax over t < key_len[b] of scale * q . K for head
 *                      (l_k, h_k) of slot b, and 0 for t >= key_len[b]
 *   mean[b][t]       = average of weights[b][k][t] over the nsel heads
 *
 *   Q         device fp32 [B][L][H][dh] (the decode step's queries), 16-byte aligned.
 *   heads_lh  HOST int32 [nsel][2]: (layer, head) pairs, checked against L and H.
 *   nsel      1 .. 64.
 *   weights   device fp32 [B][nsel][T] (written completely).
 *   mean      device fp32 [B][T], or NULL to skip it.
 * Errors as for cxa_decode, and CXA_EINVAL for bad nsel or head indices.
 * One kernel, launched like cxa_decode's (programmatic dependent launch: the
 * cache and key_len are read before the preceding kernel has finished, Q and
 * the outputs only after). Out-of-range key_len values are clamped to [0, T].
 */
CXA_API int cxa_alignment_weights(const cxa_cache* c, const float* Q, const int* key_len,
                                  const int* heads_lh, int nsel, float* weights, float* mean,
                                  float scale, void* stream);

/*
 * Decode layers [l0, l0 + nl) only: the per-layer form a real decoder calls
 * between its other sub-layers (the trace page's decoder body interleaves
 * cross_attn with the self-attention and MLP of each layer).
 *
 *   Q, out   device fp32 [B][nl][H][dh]: row (b, i, h) is layer l0 + i.
 *   workspace  at least cxa_decode_workspace_bytes(B, T, nl, H, dh) bytes.
 * Otherwise as cxa_decode; CXA_EINVAL unless 0 <= l0 and l0 + nl <= L.
 */
CXA_API int cxa_decode_layers(const cxa_cache* c, int l0, int nl, const float* Q, const int* key_len,
                              float* out, float scale, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * The cross-attention block of one decoder layer for one decode step, in place
 * on the decoder's residual stream x ("Whisper: Trace One Encoder Tensor into
 * Every Decoder Layer", "The concept": Q_l = decoder_hidden_l x WQ_l, and the
 * decoder body's cross_attn_norm -> cross_q_proj -> cross_attn -> cross_out_proj):
 *
 *   h = LayerNorm(x[b]) over d     (biased variance, ln_eps; ln_gamma/ln_beta
 *                                   may be NULL for 1 / 0)
 *   q = h x WQ + bQ                (bQ may be NULL)
 *   a = attention of q over layer `layer`'s cached K/V (as cxa_decode_layers)
 *   x[b] = x[b] + a x WO + bO      (bO may be NULL)
 *
 *   x        device fp32 [B][d], 16-byte aligned, read and overwritten.
 *   WQ, WO   device fp32 [d][d] indexed (d_in, d_out), like WK and WV; 16-byte
 *            aligned. d must be a multiple of 32 and at most 1280.
 *   ln_gamma, ln_beta, bQ, bO  device fp32 [d].
 *   workspace  at least cxa_cross_block_workspace_bytes(B, T, L, H, dh) bytes,
 *            256-byte aligned (decode scratch, q and a), counters zero as for
 *            cxa_decode.
 * Errors as for cxa_decode, and CXA_EINVAL for a layer out of range.
 */
CXA_API size_t cxa_cross_block_workspace_bytes(int B, int T, int L, int H, int dh);

CXA_API int cxa_cross_block(const cxa_cache* c, int layer, float* x, const float* ln_gamma,
                            const float* ln_beta, float ln_eps, const float* WQ, const float* bQ,
                            const float* WO, const float* bO, const int* key_len, float scale,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Mark slot b (or every slot when b == -1) not ready: installing new encoder
 * memory invalidates the projection cache by flag ("View 3": encoder_kv_ready = 0;
 * the circuit's invalidation trigger is an encoder memory update). Host only,
 * no device work. Returns CXA_EINVAL for a slot out of range.
 */
CXA_API int cxa_invalidate(cxa_cache* c, int b);

/* 1 if slot b is ready, 0 if not, CXA_EINVAL for a bad slot or descriptor. */
CXA_API int cxa_is_ready(const cxa_cache* c, int b);

/* Static name of a status code. */
CXA_API const char* cxa_strerror(int code);

/* Detail of the calling thread's last failed call ("" if none). */
CXA_API const char* cxa_last_error_message(void);

/* Number of kernels this library has launched in this process. */
CXA_API unsigned long long cxa_launch_count(void);

/*
 * Read the device-side status word of the current device: 0, or CXA_ETIMEOUT
 * when a kernel's bounded wait expired since the word was last cleared (the
 * kernel then skipped its remaining work). Synchronises the device. clear != 0
 * resets the word. Returns CXA_ECUDA if the word cannot be read. After a
 * timeout, the decode workspace's counters must be zeroed again before reuse.
 */
CXA_API int cxa_device_status(int clear);

/*
 * Which kernel shape runs a one-query decode (cxa_decode, cxa_decode_layers,
 * cxa_decode_shared with nq = 1, cxa_decode_noalloc). Both compute the same
 * result within the decode tolerance; they differ in speed:
 *
 *   CXA_DECODE_STREAM  the persistent split-T kernel: every valid 64-key chunk of
 *                      every row numbered densely and dealt out in equal ranges to
 *                      two CTAs per SM, split rows merged by the last arriving CTA.
 *                      Bandwidth-optimal for long streams (batched memories).
 *   CXA_DECODE_ROWS    the latency shape: a cluster of C CTAs per (slot, layer,
 *                      head) row (C = SMs / rows, at most 8), every warp issuing its
 *                      own copies, the cluster's states merged over distributed
 *                      shared memory; no workspace is touched. Taken only when the
 *                      rows fit on the SMs (rows <= SM count).
 *   CXA_DECODE_AUTO    (default) the latency shape when the rows fit and the stream
 *                      is short (rows x ceil(T / 64) <= 8 x SM count: one or a few
 *                      memories), the persistent kernel otherwise.
 *
 * Process-wide; returns CXA_EINVAL for an unknown value. Host only.
 */
#define CXA_DECODE_AUTO   0
#define CXA_DECODE_STREAM 1
#define CXA_DECODE_ROWS   2

CXA_API int cxa_set_decode_policy(int policy);

/*
 * Which kernel shape runs the populate GEMM (cxa_populate, cxa_populate_packed).
 * Both write bit-identical caches; they differ in speed:
 *
 *   CXA_POPULATE_PAIR    a cluster of two CTAs per 256 x 256 output tile sharing one
 *                        tensor-core MMA (tcgen05 cta_group::2): each CTA holds 128
 *                        rows of E and 128 columns of the packed weights per k-block,
 *                        so an SM loads a third less operand data per product than
 *                        with one CTA per tile. A populate returns CXA_EINVAL when
 *                        pairs cannot be resident on the device.
 *   CXA_POPULATE_SINGLE  one CTA per 128 x 256 output tile.
 *   CXA_POPULATE_AUTO    (default) pairs when the device can hold them and the GEMM
 *                        has at least 4 x (SM count) one-CTA tiles (nb x ceil(T / 128)
 *                        x ceil(2 L d / 256)); one CTA per tile for smaller GEMMs,
 *                        where the pairs' larger tiles leave more SMs idle.
 *
 * Process-wide; returns CXA_EINVAL for an unknown value. Host only.
 */
#define CXA_POPULATE_AUTO   0
#define CXA_POPULATE_PAIR   1
#define CXA_POPULATE_SINGLE 2

CXA_API int cxa_set_populate_policy(int policy);

/*
 * Failure-detection self-test (no counterpart in the source pages). Enqueues on
 * `stream` one kernel whose single waiting thread waits, through the same bounded
 * wait every kernel of this library uses, on a barrier that nothing completes;
 * after limit_us microseconds (1 .. 1000000) the wait gives up, the kernel sets
 * the device status word and returns, and cxa_device_status then reports
 * CXA_ETIMEOUT. Nothing faults or hangs, and the context stays usable. Returns
 * CXA_EINVAL for a limit outside that range, CXA_ECUDA if the launch fails.
 */
CXA_API int cxa_selftest_wait_timeout(unsigned int limit_us, void* stream);

/*
 * Allocation-free decode (no counterpart in the source pages: an addition of
 * this library for callers that cannot allocate device memory).
 *
 * Some callers cannot call cudaMalloc or any allocating routine: a host
 * framework that has handed all device memory to its own pool allocator, or a
 * serving loop that must not take the device-wide synchronisation and latency
 * a fresh allocation can bring. They still own Q, key_len, out and the cache,
 * but have nowhere to put the decode scratch. cxa_decode_noalloc runs the same
 * kernel as cxa_decode with its scratch (split-T partials and per-row arrival
 * counters) in a fixed array that lives in libcxa's device module: every GPU
 * that loads the library holds CXA_NOALLOC_SCRATCH_BYTES of it until the
 * process exits.
 *
 * Arguments and results are those of cxa_decode without the workspace (a short
 * stream that cxa_decode would run on the cluster-per-row kernel, which needs no
 * scratch, runs there too and leaves the array alone). The call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine. Geometry whose scratch, cxa_decode_workspace_bytes(B, T, L, H, dh),
 * exceeds CXA_NOALLOC_SCRATCH_BYTES is rejected with CXA_EINVAL (and a head_dim
 * other than 64 as unsupported geometry), launching nothing.
 *
 * Set-up and clearing: the first call in a CUDA context (per device; again after
 * a device reset) looks up the array's device address with that device current
 * (cudaGetSymbolAddress) and zeroes the array with one cudaMemsetAsync on
 * `stream`; make that first call before any stream capture begins. After that,
 * no call clears anything: the decode kernel leaves the arrival counters at zero
 * whatever the geometry, so consecutive calls overlap through programmatic
 * dependent launch exactly as cxa_decode's do. A kernel whose bounded wait
 * expired may leave counters set; once cxa_device_status has reported
 * CXA_ETIMEOUT, the next call zeroes the array again before its kernel.
 *
 * All calls share the one array and it keeps the last call's contents, so calls
 * that may overlap on the GPU (different streams without ordering, or several
 * host threads) race and produce wrong results: order them on one stream.
 */
#define CXA_NOALLOC_SCRATCH_BYTES (8u << 20)

CXA_API int cxa_decode_noalloc(const cxa_cache* c, const float* Q, const int* key_len, float* out,
                               float scale, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CXA_H_ */
