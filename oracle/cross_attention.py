"""fp64 CPU oracle for encoder-decoder cross-attention: populate and decode.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import or run this module. The product path
(the CUDA library and its Python binding) never imports it and shares no code
with it: this file uses numpy only.

What it computes, and where the pages define it:

* ``populate`` -- each decoder layer l re-projects the encoder memory E with its
  own weights, ``K_l = E x WK_l`` and ``V_l = E x WV_l`` ("Whisper: Trace One
  Encoder Tensor into Every Decoder Layer", "The concept: one tensor, many
  consumers"), plus a value bias bV_l and no key bias (the key bias is
  redundant under softmax shift invariance: "Caso de estudio: WhisperKit", §2).
  The token-major GEMM rows are re-laid out head-major ("Deliberate failure:
  token-major K meets a head-major consumer": a bit-exact copy) into a
  layer-major, head-major slab per layer (the circuit's
  ``projection_cache.storage``, "The concept"; layer-5 slab offset in "View 2").
* ``decode`` -- one query row per (slot, layer, head) attends non-causally
  ("The concept", ``"causal": false``) over the valid encoder keys, with the
  call's scale 0.125 = 1/sqrt(64) applied to q.k ("View 2 -- expand one
  cross-attention operation"); padded keys are excluded, which is the exact
  limit of the additive key-padding mask, and an empty key set gives 0 by the
  clamped softmax denominator (WhisperKit case study §2 and §4).
* ``decode_shared`` -- several query rows (hypotheses) per (slot, layer, head)
  over the slot's one cache (WhisperKit case study §3, SharedSplitKVCached).
* ``decode_layers`` / ``layer_norm`` / ``cross_block`` -- the per-layer form a
  decoder calls: LayerNorm, Q projection, attention over one layer's cache, out
  projection and residual ("The concept": Q_l = decoder_hidden_l x WQ_l and the
  cross_attn_norm -> cross_q_proj -> cross_attn -> cross_out_proj operations).
* ``attention_weights`` -- the softmax rows of chosen alignment heads and their
  mean over heads, returned for word timestamps (WhisperKit case study §6).
* ``masked_blend_update`` / ``self_attention_steps`` / ``causal_full_window`` --
  the decoder's self-attention KV cache: a fixed-length cache updated by a
  one-hot masked blend (WhisperKit case study §4), one token per step, checked
  against the causal whole-window formula ("Recurrence as feeds").
* ``full_window`` -- the "whole window" formula kept as a check beside one-query
  decode ("Recurrence as feeds", "What it opened").
* ``round_bf16`` -- fp32 -> bfloat16 round to nearest even, the conversion in
  front of the bf16 populate (the Whisper-large workload: fp32 E, bf16
  tensor-core inputs) and the rounding of a bf16 cache store.

Readings where the pages are silent (each one is pinned by a test):
  WK_l is ``[d_in, d_out]`` ("E x WK_l"); head h owns columns h*dh .. h*dh+dh-1;
  a layer slab is ``[H][T][dh]``; key_len is clamped to [0, T].

Every function here is pinned by ``tests/test_oracle_pins.py`` against brute
force, closed forms, hand-computed values and the invariants the pages fix
(``populate_head`` against ``populate`` and brute force, ``rel_frobenius``
against hand-computed ratios); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

# Clamp of the softmax denominator for an empty key set (WhisperKit case study
# §2 clamps the lazy-softmax denominator; with no keys the numerator is 0 too).
DENOM_FLOOR = 1e-300


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def check_geometry(T: int, d: int, H: int, dh: int) -> None:
    """Fail closed on the geometry the compiler rejects ("View 3 -- prefill vs
    decode": a positive encoder_memory_length and num_heads * head_dim ==
    embed_dim are hard errors)."""
    if T <= 0:
        raise ValueError("encoder memory length must be positive")
    if H * dh != d:
        raise ValueError("num_heads * head_dim must equal embed_dim")


def head_major(X: np.ndarray, H: int) -> np.ndarray:
    """Token-major ``[T, d]`` rows -> head-major ``[H, T, dh]``; column j of X is
    (head j // dh, channel j % dh). A pure copy: no value changes."""
    T, d = X.shape
    dh = d // H
    out = np.empty((H, T, dh), dtype=X.dtype)
    for h in range(H):
        out[h] = X[:, h * dh:(h + 1) * dh]
    return out


def populate(E, WK, WV, bV, H: int, bK=None):
    """Project every slot's encoder memory with every layer's WK/WV.

    E: ``[B, T, d]``; WK, WV: ``[L, d, d]`` indexed (d_in, d_out); bV: ``[L, d]``;
    bK: optional ``[L, d]`` key bias, only used by the invariance pin.
    Returns Kc, Vc as fp64 ``[B, L, H, T, dh]`` (slot, layer-major, head-major).
    """
    E, WK, WV, bV = _f64(E), _f64(WK), _f64(WV), _f64(bV)
    B, T, d = E.shape
    L = WK.shape[0]
    dh = d // H
    check_geometry(T, d, H, dh)
    Kc = np.empty((B, L, H, T, dh))
    Vc = np.empty((B, L, H, T, dh))
    for b in range(B):
        for l in range(L):
            K = E[b] @ WK[l]                 # K_l = E x WK_l        [T, d]
            V = E[b] @ WV[l] + bV[l]         # V_l = E x WV_l + bV_l [T, d]
            if bK is not None:
                K = K + _f64(bK)[l]
            Kc[b, l] = head_major(K, H)
            Vc[b, l] = head_major(V, H)
    return Kc, Vc


def populate_head(E_b, WK_l, WV_l, bV_l, h: int, dh: int = 64):
    """K and V ``[T, dh]`` of one (slot, layer, head): the same projection as
    ``populate`` restricted to head h's column block, for sampled checks at
    sizes where projecting every head in fp64 would take too long."""
    E_b = _f64(E_b)
    cols = slice(h * dh, (h + 1) * dh)
    K = E_b @ _f64(WK_l)[:, cols]
    V = E_b @ _f64(WV_l)[:, cols] + _f64(bV_l)[cols]
    return K, V


def clamp_key_len(key_len, T: int) -> np.ndarray:
    return np.clip(np.asarray(key_len, dtype=np.int64), 0, T)


def attend_row(q, K, V, n: int, scale: float) -> np.ndarray:
    """One query row against the first n keys: softmax(scale * q.K^T) V.

    The max-subtraction is the usual overflow guard; it leaves the result
    unchanged (shift invariance, WhisperKit case study §2)."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    dh = q.shape[0]
    if n <= 0:
        return np.zeros(dh)
    s = scale * (K[:n] @ q)
    w = np.exp(s - s.max())
    return (w @ V[:n]) / max(w.sum(), DENOM_FLOOR)


def decode(Q, Kc, Vc, key_len, scale: float | None = None) -> np.ndarray:
    """One decode step over all slots, layers and heads.

    Q: ``[B, L, H, dh]``; Kc, Vc: ``[B, L, H, T, dh]``; key_len: ``[B]``.
    Returns out ``[B, L, H, dh]`` (one query token, head-major)."""
    Q = _f64(Q)
    B, L, H, T, dh = np.shape(Kc)
    if scale is None:
        scale = 1.0 / np.sqrt(dh)
    n = clamp_key_len(key_len, T)
    out = np.zeros((B, L, H, dh))
    for b in range(B):
        for l in range(L):
            for h in range(H):
                out[b, l, h] = attend_row(Q[b, l, h], Kc[b, l, h], Vc[b, l, h], int(n[b]), scale)
    return out


def decode_shared(Q, Kc, Vc, key_len, scale: float | None = None) -> np.ndarray:
    """nq query rows per (slot, layer, head) over the slot's one cache: the
    beam / speculative hypotheses of one window sharing its encoder memory
    ("Caso de estudio: WhisperKit", §3, SharedSplitKVCached: a batch-N query
    attending a shared batch-1 cache).

    Q: ``[B, nq, L, H, dh]``; returns out ``[B, nq, L, H, dh]``, hypothesis n of
    slot b decoded exactly as ``decode`` decodes a single query row."""
    Q = _f64(Q)
    nq = Q.shape[1]
    return np.stack([decode(Q[:, n], Kc, Vc, key_len, scale) for n in range(nq)], axis=1)


def full_window(Qblock, K, V, n: int, scale: float) -> np.ndarray:
    """All query rows at once as one matrix-softmax-matrix: ``[nq, dh]``."""
    Qblock, K, V = _f64(Qblock), _f64(K), _f64(V)
    S = scale * (Qblock @ K[:n].T)
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    P = P / P.sum(axis=1, keepdims=True)
    return P @ V[:n]


def decode_layers(Q, Kc, Vc, key_len, l0: int, scale: float | None = None) -> np.ndarray:
    """Decode of layers [l0, l0 + nl) only: Q ``[B, nl, H, dh]`` -> out of the same shape."""
    Q = _f64(Q)
    nl = Q.shape[1]
    return decode(Q, np.asarray(Kc)[:, l0:l0 + nl], np.asarray(Vc)[:, l0:l0 + nl], key_len, scale)


def layer_norm(x, gamma=None, beta=None, eps: float = 1e-5) -> np.ndarray:
    """LayerNorm over the last axis with the biased variance (the cross_attn_norm
    of the decoder body, "The concept"; the pages name the norm, its form is
    Whisper's LayerNorm)."""
    x = _f64(x)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    y = (x - mean) / np.sqrt(var + eps)
    if gamma is not None:
        y = y * _f64(gamma)
    if beta is not None:
        y = y + _f64(beta)
    return y


def cross_block(x, layer: int, Kc, Vc, key_len, WQ, WO, gamma=None, beta=None, eps: float = 1e-5,
                bQ=None, bO=None, scale: float | None = None) -> np.ndarray:
    """One decoder layer's cross-attention block for one step ("The concept":
    Q_l = decoder_hidden_l x WQ_l; cross_attn_norm -> cross_q_proj -> cross_attn
    -> cross_out_proj), with the residual add: returns the new x ``[B, d]``."""
    x = _f64(x)
    B, d = x.shape
    H = np.shape(Kc)[2]
    dh = d // H
    q = layer_norm(x, gamma, beta, eps) @ _f64(WQ)
    if bQ is not None:
        q = q + _f64(bQ)
    a = decode_layers(q.reshape(B, 1, H, dh), Kc, Vc, key_len, layer, scale).reshape(B, d)
    y = a @ _f64(WO)
    if bO is not None:
        y = y + _f64(bO)
    return x + y


def attention_weights(Q, Kc, key_len, heads, scale: float | None = None):
    """Softmax rows of the selected (layer, head) pairs ("Caso de estudio:
    WhisperKit", §6, alignment-head weights) and their mean over the heads.
    Q ``[B, L, H, dh]``; returns (weights ``[B, nsel, T]``, mean ``[B, T]``),
    zero beyond key_len."""
    Q, Kc = _f64(Q), _f64(Kc)
    B, L, H, T, dh = Kc.shape
    if scale is None:
        scale = 1.0 / np.sqrt(dh)
    n = clamp_key_len(key_len, T)
    w = np.zeros((B, len(heads), T))
    for b in range(B):
        if n[b] == 0:
            continue
        for k, (l, h) in enumerate(heads):
            s = scale * (Kc[b, l, h, :n[b]] @ Q[b, l, h])
            e = np.exp(s - s.max())
            w[b, k, :n[b]] = e / e.sum()
    return w, w.mean(axis=1)


def masked_blend_update(cache, new_row, pos):
    """One-hot masked blend of a new row into a fixed-length cache
    ("Caso de estudio: WhisperKit", §4): cache*(1 - onehot(pos)) + new*onehot(pos).
    cache ``[T, dh]``, new_row ``[dh]``; returns the updated cache (fp64)."""
    cache = _f64(cache)
    T = cache.shape[0]
    mask = np.zeros((T, 1))
    if 0 <= pos < T:
        mask[pos, 0] = 1.0
    return cache * (1.0 - mask) + _f64(new_row)[None, :] * mask


def self_attention_steps(Qs, Ks, Vs, scale: float | None = None) -> np.ndarray:
    """Token-by-token self-attention decode: step i appends key/value row i to an
    empty cache (by the masked blend) and attends positions 0 .. i.
    Qs, Ks, Vs ``[S, dh]``; returns ``[S, dh]``."""
    Qs, Ks, Vs = _f64(Qs), _f64(Ks), _f64(Vs)
    S, dh = Qs.shape
    if scale is None:
        scale = 1.0 / np.sqrt(dh)
    Kc, Vc = np.zeros((S, dh)), np.zeros((S, dh))
    out = np.zeros((S, dh))
    for i in range(S):
        Kc = masked_blend_update(Kc, Ks[i], i)
        Vc = masked_blend_update(Vc, Vs[i], i)
        out[i] = attend_row(Qs[i], Kc, Vc, i + 1, scale)
    return out


def causal_full_window(Qs, Ks, Vs, scale: float | None = None) -> np.ndarray:
    """The whole window at once with a causal mask: row i attends keys 0 .. i
    ("Recurrence as feeds": the run-the-whole-window formula kept as a check of
    one-token decode)."""
    Qs, Ks, Vs = _f64(Qs), _f64(Ks), _f64(Vs)
    S, dh = Qs.shape
    if scale is None:
        scale = 1.0 / np.sqrt(dh)
    Sc = scale * (Qs @ Ks.T)
    Sc = np.where(np.tril(np.ones((S, S), dtype=bool)), Sc, -np.inf)
    Sc = Sc - Sc.max(axis=1, keepdims=True)
    P = np.exp(Sc)
    P = P / P.sum(axis=1, keepdims=True)
    return P @ Vs


def cross_attention_from_memory(Q, E, WK, WV, bV, key_len, H: int, scale: float | None = None):
    """Decode computed by re-projecting E (no cache), for the cache-reuse pin."""
    Kc, Vc = populate(E, WK, WV, bV, H)
    return decode(Q, Kc, Vc, key_len, scale)


def round_bf16(x) -> np.ndarray:
    """fp32 values rounded to the nearest bfloat16 (8 significant bits: the fp32
    value with its 16 low fraction bits cleared), ties to the even significand.
    Written from the rounding rule: the two bf16 neighbours of x are x with its 16
    low bits cleared (toward zero) and the next bf16 away from zero; the nearer
    one is taken, the distances measured exactly in fp64 (fp32 differences are
    exact there); a tie takes the neighbour whose last kept bit is 0. Past the
    largest finite bf16 the upper neighbour is infinity, which the rule places at
    2^128 (one ulp beyond); infinities and NaNs pass through. Returns float32."""
    x32 = np.array(x, dtype=np.float32)      # a copy, of x's shape (0-d for a scalar)
    bits = x32.view(np.uint32)
    lo_bits = bits & np.uint32(0xFFFF0000)
    hi_bits = lo_bits + np.uint32(0x10000)
    xd = x32.astype(np.float64)
    special = ~np.isfinite(xd)
    with np.errstate(invalid="ignore"):
        lo = lo_bits.view(np.float32).astype(np.float64)
        hi = hi_bits.view(np.float32).astype(np.float64)
        hi_pos = np.where(np.isinf(hi), np.copysign(2.0 ** 128, xd), hi)
        d_lo = np.abs(xd - lo)
        d_hi = np.abs(hi_pos - xd)
    lo_even = ((lo_bits >> np.uint32(16)) & np.uint32(1)) == 0
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ~lo_even)
    out = np.where(take_hi, hi, lo)
    out = np.where(special, xd, out)
    return out.astype(np.float32)


def rel_frobenius(x, ref) -> float:
    """Relative Frobenius error ||x - ref||_F / ||ref||_F over all elements: the
    measure the populate tolerance is stated in (square root of the summed
    squared differences over the square root of the summed squared reference)."""
    x, ref = _f64(x), _f64(ref)
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))
