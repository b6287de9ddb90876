"""Self-attention KV cache on the GPU: cxa_cache_append + decode over positions
0 .. pos (cxa_self_attention_step), step by step without host syncs, against the
oracle's token-by-token decode (which itself equals the causal whole-window
formula). Slots start at different steps (a slot whose position is still
negative appends nothing and decodes to zeros)."""
import numpy as np
import pytest
import torch

from _gpu_common import DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, dev, host, inputs_on_device
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W
from oracle import cross_attention as O

pytestmark = pytest.mark.gpu
TOL = {"f32": DECODE_F32_MAX_ABS, "bf16": DECODE_BF16_MAX_ABS}


@pytest.fixture(scope="module", autouse=True)
def _lib(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.synchronize()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_token_by_token_steps(cache_dtype):
    B, L, H, T, S = 4, 2, 3, 448, 70
    delay = np.array([0, 3, 17, 69])                 # slot b begins at step delay[b]
    c = cxa.CrossAttentionCache(B, T, L, H, 64, cache_dtype)
    Qs, Ks, Vs = _rand((S, B, L, H, 64), 1), _rand((S, B, L, H, 64), 2), _rand((S, B, L, H, 64), 3)
    if cache_dtype == "bf16":                         # the cache stores bf16: compare on the stored values
        Ks, Vs = W.bf16_round(Ks), W.bf16_round(Vs)
    pos = [dev((s - delay).astype(np.int32), torch.int32) for s in range(S)]
    Qd, Kd, Vd = [dev(q) for q in Qs], [dev(k) for k in Ks], [dev(v) for v in Vs]
    outs = [torch.empty((B, L, H, 64), device="cuda") for _ in range(S)]
    torch.cuda.synchronize()
    for s in range(S):
        c.self_attention_step(pos[s], Qd[s], Kd[s], Vd[s], out=outs[s])
    torch.cuda.synchronize()
    got = np.stack([host(o) for o in outs])
    for b in range(B):
        n = S - delay[b]
        assert np.all(got[:delay[b], b] == 0.0)
        for l in range(L):
            for h in range(H):
                ref = O.self_attention_steps(Qs[delay[b]:, b, l, h], Ks[delay[b]:, b, l, h], Vs[delay[b]:, b, l, h])
                assert np.abs(got[delay[b]:, b, l, h] - ref).max() <= TOL[cache_dtype]
        # the cache holds exactly the appended rows
        assert np.array_equal(host(c.Kc[b, :, :, :n]), np.moveaxis(Ks[delay[b]:, b], 0, 2).astype(np.float64))


def test_end_of_cache_and_out_of_range_positions():
    B, L, H, T = 3, 1, 2, 448
    c = cxa.CrossAttentionCache(B, T, L, H, 64, "f32")
    c.Kc.zero_()
    c.Vc.zero_()
    K0, V0 = _rand((B, L, H, 64), 5), _rand((B, L, H, 64), 6)
    c.append(dev(np.array([447, 448, -1], np.int32), torch.int32), dev(K0), dev(V0))
    torch.cuda.synchronize()
    assert np.array_equal(host(c.Kc[0, :, :, 447]), K0[0].astype(np.float64))
    assert not host(c.Kc[1]).any() and not host(c.Kc[2]).any()     # nothing written out of range
    # decode with key_len = pos + 1 beyond T clamps to T
    Q = _rand((B, L, H, 64), 7)
    out = host(c.self_attention_step(dev(np.array([447, 500, 0], np.int32), torch.int32), dev(Q), dev(K0), dev(V0)))
    ref = O.decode(Q, host(c.Kc), host(c.Vc), np.array([448, 500 + 1, 1]))
    assert np.abs(out - ref).max() <= DECODE_F32_MAX_ABS


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_long_sequence_rewind_and_interleaved_decodes(cache_dtype):
    """300 steps, then both slots start a new sequence at position 0 for 160 more, with
    a cross-attention decode (a kernel that lets its successor start at once) launched
    between every two steps and no host syncs. A step streams the rows below pos - 1
    before the previous kernel has finished: every output must still match the
    oracle's token-by-token decode of its own sequence."""
    from _gpu_common import cache_for, inputs_on_device
    B, L, H, T, S1, S2 = 2, 1, 2, 448, 300, 160
    c = cxa.CrossAttentionCache(B, T, L, H, 64, cache_dtype)
    w = W.custom("sa_cross", B=B, T=200, d=128, L=L, H=H, index=980)
    d, _ = inputs_on_device(w)
    cross = cache_for(w, "f32")
    cross.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Qc = dev(W.make_Q(w, 1))
    seqs = []
    for k, S in enumerate((S1, S2)):
        Qs, Ks, Vs = _rand((S, B, L, H, 64), 20 + k), _rand((S, B, L, H, 64), 30 + k), _rand((S, B, L, H, 64), 40 + k)
        if cache_dtype == "bf16":
            Ks, Vs = W.bf16_round(Ks), W.bf16_round(Vs)
        seqs.append((Qs, Ks, Vs))
    outs = []
    torch.cuda.synchronize()
    for Qs, Ks, Vs in seqs:
        S = Qs.shape[0]
        pos = [dev(np.full(B, s, np.int32), torch.int32) for s in range(S)]
        Qd, Kd, Vd = [dev(q) for q in Qs], [dev(x) for x in Ks], [dev(x) for x in Vs]
        o = [torch.empty((B, L, H, 64), device="cuda") for _ in range(S)]
        for s in range(S):
            c.self_attention_step(pos[s], Qd[s], Kd[s], Vd[s], out=o[s])
            cross.decode(Qc, d["key_len"])
        outs.append(o)
    torch.cuda.synchronize()
    for (Qs, Ks, Vs), o in zip(seqs, outs):
        got = np.stack([host(x) for x in o])
        for b in range(B):
            for l in range(L):
                for h in range(H):
                    ref = O.self_attention_steps(Qs[:, b, l, h], Ks[:, b, l, h], Vs[:, b, l, h])
                    assert np.abs(got[:, b, l, h] - ref).max() <= TOL[cache_dtype]


def test_append_and_populate_refuse_each_others_cache():
    """A populated (cross-attention) cache refuses appends, which would mark its
    invalidated slots ready again; a self-attention cache refuses populate."""
    w = W.custom("roles", B=2, T=64, d=128, L=1, H=2, index=942)
    d, _ = inputs_on_device(w)
    cross = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, 64, "f32")
    cross.populate(d["E"], d["WK"], d["WV"], d["bV"])
    cross.invalidate(1)
    pos = dev(np.array([3, 4], np.int32), torch.int32)
    rows = dev(np.zeros((w.B, w.L, w.H, 64), np.float32))
    launches = cxa.cxa_launch_count()
    assert cxa.cxa_cache_append(cross.handle, pos, rows, rows) == cxa.CXA_EINVAL
    out = torch.empty_like(rows)
    assert cxa.cxa_self_attention_step(cross.handle, pos, rows, rows, rows, out, 0.0, cross.decode_ws,
                                       cross.decode_ws_bytes) == cxa.CXA_EINVAL
    assert cxa.cxa_launch_count() == launches
    assert not cross.is_ready(1)
    selfc = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, 64, "f32")
    selfc.append(pos, rows, rows)
    torch.cuda.synchronize()
    assert selfc.is_ready(0) and selfc.is_ready(1)
    ws = selfc.populate_workspace(cxa.CXA_F32)
    rc = cxa.cxa_populate(selfc.handle, 0, w.B, d["E"], d["WK"], d["WV"], d["bV"], w.T, w.d, w.L, w.H, cxa.CXA_F32,
                          ws, ws.numel())
    assert rc == cxa.CXA_EINVAL
