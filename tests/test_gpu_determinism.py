"""Repeatability: the same inputs give bit-identical outputs call after call. Split
rows are merged from their segments' partial states in segment order, whichever
CTA arrives last, and no kernel accumulates with atomics, so repeated launches
(back to back, without host syncs in between) must agree to the last bit."""
import numpy as np
import pytest
import torch

from _gpu_common import cache_for, decode_policy, dev, inputs_on_device, populate_policy
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.synchronize()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def _batched(cache_dtype, index):
    w = W.custom("repeat", B=16, T=1500, d=512, L=6, H=8, ragged=True, index=index)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    return w, d, h, c


@pytest.mark.parametrize("shape", ["stream", "rows", "auto"])
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_decode_repeats_bit_for_bit(shape, cache_dtype):
    w, d, _, c = _batched(cache_dtype, 970)
    Q = dev(W.make_Q(w, 0))
    with decode_policy(shape):
        outs = [c.decode(Q, d["key_len"], out=torch.empty_like(Q)) for _ in range(5)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("cache_dtype,nq", [("f32", 5), ("f32", 8), ("bf16", 8), ("bf16", 16)])
def test_shared_decode_repeats_bit_for_bit(cache_dtype, nq):
    w, d, _, c = _batched(cache_dtype, 971)
    Q = dev(np.random.default_rng(972).standard_normal((w.B, nq, w.L, w.H, 64)).astype(np.float32))
    outs = [c.decode_shared(Q, d["key_len"], out=torch.empty_like(Q)) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("shape", ["pair", "single"])
def test_populate_repeats_bit_for_bit(shape):
    w = W.custom("repeat_pop", B=16, T=1500, d=512, L=6, H=8, ragged=True, index=973)
    d, _ = inputs_on_device(w)
    caches = []
    with populate_policy(shape):
        for _ in range(2):
            c = cache_for(w, "f32")
            c.populate(d["E"], d["WK"], d["WV"], d["bV"])
            caches.append(c)
    torch.cuda.synchronize()
    assert torch.equal(caches[0].Kc, caches[1].Kc) and torch.equal(caches[0].Vc, caches[1].Vc)


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_cross_block_and_alignment_repeat_bit_for_bit(cache_dtype):
    w, d, _, c = _batched(cache_dtype, 974)
    rng = np.random.default_rng(975)
    WQ = dev((rng.standard_normal((w.d, w.d)) * w.d ** -0.5).astype(np.float32))
    WO = dev((rng.standard_normal((w.d, w.d)) * w.d ** -0.5).astype(np.float32))
    x0 = dev(rng.standard_normal((w.B, w.d)).astype(np.float32))
    xs = [x0.clone() for _ in range(3)]
    for x in xs:
        c.cross_block(2, x, WQ, WO, d["key_len"])
    Q = dev(W.make_Q(w, 1))
    heads = [(0, 1), (2, 5), (4, 4), (5, 7)]
    al = [c.alignment_weights(Q, d["key_len"], heads) for _ in range(3)]
    torch.cuda.synchronize()
    for x in xs[1:]:
        assert torch.equal(x, xs[0])
    for wt, m in al[1:]:
        assert torch.equal(wt, al[0][0]) and torch.equal(m, al[0][1])


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_self_attention_steps_repeat_bit_for_bit(cache_dtype):
    B, L, H, T, S = 16, 6, 8, 448, 24
    rng = np.random.default_rng(976)
    Qs, Ks, Vs = (dev(rng.standard_normal((S, B, L, H, 64)).astype(np.float32)) for _ in range(3))
    pos = [dev(np.full(B, 200 + s, np.int32), torch.int32) for s in range(S)]
    results = []
    for _ in range(2):
        c = cxa.CrossAttentionCache(B, T, L, H, 64, cache_dtype)
        c.Kc.zero_()
        c.Vc.zero_()
        outs = [torch.empty((B, L, H, 64), device="cuda") for _ in range(S)]
        for s in range(S):
            c.self_attention_step(pos[s], Qs[s], Ks[s], Vs[s], out=outs[s])
        results.append((outs, c))
    torch.cuda.synchronize()
    for a, b in zip(results[0][0], results[1][0]):
        assert torch.equal(a, b)
    assert torch.equal(results[0][1].Kc, results[1][1].Kc)
