"""Seeded synthetic inputs for Whisper-shaped cross-attention workloads.

This module only draws random tensors and describes workload shapes; it holds
none of the cross-attention arithmetic, so both the CUDA path (through the
binding) and the fp64 oracle can be fed from it without sharing any of the
method's code.

Shapes follow the Whisper dimensions on the pages: encoder memory E is a
token-major ``[T_enc, d]`` grid (Whisper Base ``[1500, 512]``, "Whisper: Trace
One Encoder Tensor into Every Decoder Layer", "The concept: one tensor, many
consumers"); each decoder layer owns ``WK_l``/``WV_l`` of shape ``[d_in, d_out]``
and a value bias ``bV_l`` (the key bias is dropped as redundant, WhisperKit case
study §2); one query row per (batch, layer, head) per decode step.

Seeds: every tensor draws from ``numpy.random.default_rng(seed)`` (PCG64) with
``seed = 1_000_000 * workload.index + 1000 * tensor_id + sub`` where ``sub`` is
the batch slot (E) or the decode step (Q). Per-slot and per-step streams are
independent, so a single slot or step can be regenerated without the rest.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple

import numpy as np

# tensor ids inside a workload's seed space
_T_E, _T_WK, _T_WV, _T_BV, _T_Q, _T_KEYLEN = 0, 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Workload:
    name: str
    index: int              # seed namespace
    B: int                  # independent encoder memories (batch slots)
    T: int                  # encoder length T_enc
    d: int                  # model width
    L: int                  # decoder layers
    H: int                  # heads
    steps: int              # decode steps per window
    in_dtype: str = "f32"   # "f32" -> TF32 tensor-core populate, "bf16" -> bf16 populate
    cache_dtypes: Tuple[str, ...] = ("f32",)
    ragged: bool = False    # key_len_b ~ U{T/3 .. T}, padded E rows zeroed
    dh: int = 64
    e_std: float = 1.0
    w_std: float = field(default=0.0)   # 0 -> 1/sqrt(d)
    bv_std: float = 0.02

    @property
    def weight_std(self) -> float:
        return self.w_std if self.w_std > 0 else float(1.0 / np.sqrt(self.d))

    @property
    def scale(self) -> float:
        return float(1.0 / np.sqrt(self.dh))


WORKLOADS = {
    # Whisper-tiny dims: 4 layers, 6 heads x 64; one populate + one decode step.
    "tiny": Workload("tiny", 0, B=1, T=1500, d=384, L=4, H=6, steps=1),
    # Whisper-Base dims: 6 layers, 8 heads x 64; 64 decode steps on a reused cache.
    "base": Workload("base", 1, B=1, T=1500, d=512, L=6, H=8, steps=64),
    # Batched Whisper-Base: 16 memories, ragged key_len ~ U{500..1500}.
    "batched_base": Workload("batched_base", 2, B=16, T=1500, d=512, L=6, H=8, steps=128,
                             cache_dtypes=("f32", "bf16"), ragged=True),
    # Whisper-large dims: 32 layers, 20 heads x 64, batch 8, bf16 populate and cache.
    "large": Workload("large", 3, B=8, T=1500, d=1280, L=32, H=20, steps=256,
                      in_dtype="bf16", cache_dtypes=("bf16",)),
}

# Decode bandwidth sweep: d=512, 8x64 heads, 6 layers, E and W ~ N(0, 1/d).
SWEEP_T = (256, 1500, 4096, 16384, 32768)
SWEEP_B = (1, 4, 16, 64)


def sweep_workload(T: int, B: int) -> Workload:
    return Workload(f"sweep_T{T}_B{B}", 100 + SWEEP_T.index(T) * 10 + SWEEP_B.index(B),
                    B=B, T=T, d=512, L=6, H=8, steps=100, cache_dtypes=("f32", "bf16"),
                    e_std=float(1.0 / np.sqrt(512)))


def custom(name: str, B: int, T: int, d: int, L: int, H: int, *, index: int = 900,
           steps: int = 1, in_dtype: str = "f32", ragged: bool = False, dh: int = 64,
           **kw) -> Workload:
    """A workload of arbitrary small shape for tests (same distributions as Base)."""
    return Workload(name, index, B=B, T=T, d=d, L=L, H=H, steps=steps, in_dtype=in_dtype,
                    ragged=ragged, dh=dh, **kw)


def _seed(w: Workload, tensor: int, sub: int = 0) -> int:
    return 1_000_000 * w.index + 1000 * tensor + sub


def _normal(seed: int, shape, std: float) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def make_key_len(w: Workload) -> np.ndarray:
    """int32 [B]: T for every slot, or U{T/3 .. T} inclusive for ragged workloads
    (500..1500 at T = 1500)."""
    if not w.ragged:
        return np.full((w.B,), w.T, dtype=np.int32)
    rng = np.random.default_rng(_seed(w, _T_KEYLEN))
    lo = max(1, w.T // 3)
    return rng.integers(lo, w.T, size=w.B, endpoint=True).astype(np.int32)


def make_E(w: Workload, b: int, key_len: np.ndarray | None = None) -> np.ndarray:
    """float32 [T, d] encoder memory of slot b; rows t >= key_len[b] are zero padding."""
    E = _normal(_seed(w, _T_E, b), (w.T, w.d), w.e_std)
    if w.ragged:
        kl = make_key_len(w) if key_len is None else key_len
        E[int(kl[b]):] = 0.0
    return maybe_bf16(w, E)


def make_E_all(w: Workload) -> np.ndarray:
    kl = make_key_len(w)
    return np.stack([make_E(w, b, kl) for b in range(w.B)])


def make_weights(w: Workload):
    """WK, WV float32 [L, d, d] as (d_in, d_out); bV float32 [L, d]."""
    WK = maybe_bf16(w, _normal(_seed(w, _T_WK), (w.L, w.d, w.d), w.weight_std))
    WV = maybe_bf16(w, _normal(_seed(w, _T_WV), (w.L, w.d, w.d), w.weight_std))
    bV = _normal(_seed(w, _T_BV), (w.L, w.d), w.bv_std)
    return WK, WV, bV


def make_Q(w: Workload, step: int) -> np.ndarray:
    """float32 [B, L, H, dh]: one fresh query row per (slot, layer, head) at a step."""
    return _normal(_seed(w, _T_Q, step), (w.B, w.L, w.H, w.dh), 1.0)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of float32 values, round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 values rounded (RN-even) to the nearest bf16 value."""
    return bf16_to_f32(bf16_bits(x))


def maybe_bf16(w: Workload, x: np.ndarray) -> np.ndarray:
    """Inputs of a bf16-input workload are drawn in fp32 and rounded to bf16, so the
    GPU (fed bf16) and the oracle (fed the same values in fp64) see identical data."""
    return bf16_round(x) if w.in_dtype == "bf16" else x


__all__ = ["Workload", "WORKLOADS", "SWEEP_T", "SWEEP_B", "sweep_workload", "custom",
           "make_key_len", "make_E", "make_E_all", "make_weights", "make_Q",
           "bf16_bits", "bf16_to_f32", "bf16_round", "maybe_bf16", "replace"]
