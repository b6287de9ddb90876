"""The populate parity gates themselves, on the CPU: a GEMM that does what the
tensor-core path does (fp32 operands read as TF32 -- E truncated, W rounded to
nearest -- or bf16 operands, fp32 accumulation, fp32 or bf16-RNE stores) must
pass the element-wise and per-block gates of ``_gpu_common.check_populate``,
and plausible mistakes (one (t, head) row taken from the next token, the value
bias dropped on one head, a block's largest element 2 % off) must fail them. This shows the
gates are tight enough to catch what a norm over a whole cache misses."""
import numpy as np
import pytest

from _gpu_common import check_populate
from encoder_decoder_speech_gb300 import workloads as W


def _tf32_trunc(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u & np.uint32(0xFFFFE000)).view(np.float32)


def _tf32_rna(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def _emulated_populate(E, WK, WV, bV, H, in_dtype, cache_dtype):
    """[B, L, H, T, dh] K/V as the tensor-core path computes them (in fp32)."""
    B, T, d = E.shape
    L, dh = WK.shape[0], d // H
    Ea = _tf32_trunc(E) if in_dtype == "f32" else E.astype(np.float32)
    K = np.empty((B, L, H, T, dh), np.float32)
    V = np.empty((B, L, H, T, dh), np.float32)
    for l in range(L):
        wk = _tf32_rna(WK[l]) if in_dtype == "f32" else WK[l].astype(np.float32)
        wv = _tf32_rna(WV[l]) if in_dtype == "f32" else WV[l].astype(np.float32)
        for b in range(B):
            k = Ea[b] @ wk
            v = Ea[b] @ wv + bV[l].astype(np.float32)
            K[b, l] = k.reshape(T, H, dh).transpose(1, 0, 2)
            V[b, l] = v.reshape(T, H, dh).transpose(1, 0, 2)
    if cache_dtype == "bf16":
        K, V = W.bf16_round(K), W.bf16_round(V)
    return K.astype(np.float64), V.astype(np.float64)


def _case(in_dtype):
    w = W.custom("gates", B=2, T=200, d=256, L=2, H=4, in_dtype=in_dtype, index=930)
    E = W.make_E_all(w)
    WK, WV, bV = W.make_weights(w)
    return w, E, WK, WV, bV


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_emulated_tensor_core_populate_passes(in_dtype, cache_dtype):
    w, E, WK, WV, bV = _case(in_dtype)
    Kg, Vg = _emulated_populate(E, WK, WV, bV, w.H, in_dtype, cache_dtype)
    fk, fv, worst = check_populate(Kg, Vg, E, WK, WV, bV, w.H, in_dtype, cache_dtype, "emulated")
    assert fk < 2e-3 and fv < 2e-3 and worst < 5e-3


def _plant(Kg, Vg, kind):
    Kg, Vg = Kg.copy(), Vg.copy()
    if kind == "next_token_row":
        Kg[1, 1, 2, 57] = Kg[1, 1, 2, 58]
    elif kind == "value_bias_dropped_on_one_head":
        return Kg, Vg, ("bias", 0, 1, 3)
    elif kind == "largest_element_2pct":
        blk = Vg[0, 0, 1]
        blk[np.unravel_index(np.abs(blk).argmax(), blk.shape)] *= 1.02
    return Kg, Vg, None


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["next_token_row", "value_bias_dropped_on_one_head", "largest_element_2pct"])
def test_planted_populate_mistakes_fail_the_gates(kind, cache_dtype):
    w, E, WK, WV, bV = _case("f32")
    Kg, Vg = _emulated_populate(E, WK, WV, bV, w.H, "f32", cache_dtype)
    Kg, Vg, extra = _plant(Kg, Vg, kind)
    if extra is not None:                           # drop bV on head 3 of layer 1, slot 0
        _, b, l, h = extra
        Vg[b, l, h] -= bV[l, h * 64:(h + 1) * 64][None, :]
    with pytest.raises(AssertionError):
        check_populate(Kg, Vg, E, WK, WV, bV, w.H, "f32", cache_dtype, "planted")
