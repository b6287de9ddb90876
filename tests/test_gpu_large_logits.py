"""Decode with extreme logits, checked against the oracle on the very cache the
GPU holds: in every (slot, layer, head) row one key is planted along that row's
query, so its score is about +200 and the softmax row is one-hot up to e^-190.
The planted key sits first in the row, last among its valid keys, or in between,
so the running maximum moves at the start, at the very end or in the middle of a
row (and of a row split across CTAs, whose segments then merge with maxima
hundreds apart). Every other key keeps its ordinary score. A kernel that lets a
stale maximum through, drops a rescale or mis-weights a segment returns a mix of
V rows instead of the planted key's row."""
import numpy as np
import pytest
import torch

from _gpu_common import DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, cache_for, decode_policy, dev, host, inputs_on_device
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W
from oracle import cross_attention as O

pytestmark = pytest.mark.gpu

TOL = {"f32": DECODE_F32_MAX_ABS, "bf16": DECODE_BF16_MAX_ABS}
SPIKE_SCORE = 200.0   # scale * q.k of the planted key (natural-log units)


@pytest.fixture(scope="module", autouse=True)
def _lib(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.synchronize()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def _plant(c, q_rows, key_len, layers=None):
    """Set one key per (slot, layer, head) row of the cache (of the given layers,
    all by default) to a multiple of that row's query q_rows [B, L, H, 64], scaled
    so that 0.125 * q.k = SPIKE_SCORE. Returns the planted positions [B, L, H]
    (-1 where nothing was planted)."""
    B, L, H = q_rows.shape[:3]
    pos = np.full((B, L, H), -1, dtype=np.int64)
    Kc = c.Kc
    for b in range(B):
        n = int(min(max(key_len[b], 0), c.T))
        if n == 0:
            continue
        for l in range(L) if layers is None else layers:
            for h in range(H):
                choice = (l * H + h) % 3
                t = 0 if choice == 0 else (n - 1 if choice == 1 else (b * 31 + l * 7 + h * 3) % n)
                q = q_rows[b, l, h].astype(np.float64)
                alpha = SPIKE_SCORE / (0.125 * float(q @ q))
                Kc[b, l, h, t] = torch.from_numpy((alpha * q).astype(np.float32)).to(Kc.device, Kc.dtype)
                pos[b, l, h] = t
    return pos


def _workload(index):
    return W.custom("large_logits", B=5, T=900, d=256, L=2, H=4, ragged=True, index=index)


@pytest.mark.parametrize("shape", ["stream", "rows"])
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_decode_one_hot_rows(shape, cache_dtype):
    w = _workload(950)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Qh = W.make_Q(w, 0)
    pos = _plant(c, Qh, h["key_len"])
    torch.cuda.synchronize()
    K, V = host(c.Kc), host(c.Vc)
    with decode_policy(shape):
        out = host(c.decode(dev(Qh), d["key_len"]))
    ref = O.decode(Qh, K, V, h["key_len"])
    # precondition: the oracle's rows are the planted keys' V rows
    for b in range(w.B):
        for l in range(w.L):
            for hh in range(w.H):
                if pos[b, l, hh] >= 0:
                    assert np.abs(ref[b, l, hh] - V[b, l, hh, pos[b, l, hh]]).max() < 1e-9
    assert np.isfinite(out).all()
    assert np.abs(out - ref).max() <= TOL[cache_dtype]


@pytest.mark.parametrize("cache_dtype,nq", [("f32", 2), ("f32", 5), ("f32", 8), ("bf16", 2), ("bf16", 8)])
def test_shared_decode_one_hot_rows(cache_dtype, nq):
    """The key of each row is planted along its first hypothesis' query; the other
    hypotheses see that key at a large score of either sign."""
    w = _workload(951)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    rng = np.random.default_rng(952 + nq)
    Q = rng.standard_normal((w.B, nq, w.L, w.H, 64)).astype(np.float32)
    _plant(c, Q[:, 0], h["key_len"])
    torch.cuda.synchronize()
    K, V = host(c.Kc), host(c.Vc)
    out = host(c.decode_shared(dev(Q), d["key_len"]))
    ref = O.decode_shared(Q, K, V, h["key_len"])
    assert np.isfinite(out).all()
    assert np.abs(out - ref).max() <= TOL[cache_dtype]


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_alignment_weights_one_hot_rows(cache_dtype):
    """The alignment-head rows of planted keys are one-hot at the planted position
    (the clusters' partial maxima then differ by hundreds between CTAs), and their
    head mean is the mean of those one-hot rows."""
    w = W.custom("large_logits_align", B=16, T=1500, d=512, L=6, H=8, ragged=True, index=953)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Qh = W.make_Q(w, 0)
    pos = _plant(c, Qh, h["key_len"])
    torch.cuda.synchronize()
    heads = [(0, 0), (1, 5), (2, 2), (3, 7), (4, 1), (5, 4)]
    wt, mean = c.alignment_weights(dev(Qh), d["key_len"], heads)
    wt, mean = host(wt), host(mean)
    ref_w, ref_m = O.attention_weights(Qh, host(c.Kc), h["key_len"], heads)
    for b in range(w.B):
        for k, (l, hh) in enumerate(heads):
            if pos[b, l, hh] >= 0:
                assert abs(ref_w[b, k, pos[b, l, hh]] - 1.0) < 1e-9
    assert np.isfinite(wt).all() and np.isfinite(mean).all()
    assert np.abs(wt - ref_w).max() <= 1e-5
    assert np.abs(mean - ref_m).max() <= 1e-5


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H", [(16, 8), (5, 4)])
def test_cross_block_one_hot_rows(cache_dtype, B, H):
    """The block's attention (LayerNorm, query projection, attention, out projection):
    keys planted along the projected queries LayerNorm(x) WQ + bQ. Batched-Base
    width takes the two-launch form (its clusters do not all fit), the small width
    the one-launch form."""
    d_model = 64 * H
    w = W.custom("large_logits_block", B=B, T=1500 if B == 16 else 400, d=d_model, L=2, H=H, ragged=True,
                 index=954)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    rng = np.random.default_rng(955)
    p = {"WQ": rng.standard_normal((d_model, d_model)) * d_model ** -0.5,
         "WO": rng.standard_normal((d_model, d_model)) * d_model ** -0.5,
         "gamma": 1.0 + 0.1 * rng.standard_normal(d_model), "beta": 0.1 * rng.standard_normal(d_model),
         "bQ": 0.02 * rng.standard_normal(d_model), "bO": 0.02 * rng.standard_normal(d_model)}
    p = {k: v.astype(np.float32) for k, v in p.items()}
    x0 = rng.standard_normal((B, d_model)).astype(np.float32)
    layer = 1
    q = (O.layer_norm(x0, p["gamma"], p["beta"], 1e-5) @ p["WQ"].astype(np.float64) + p["bQ"]).reshape(B, H, 64)
    q_rows = np.zeros((B, w.L, H, 64), np.float32)
    q_rows[:, layer] = q
    pos = _plant(c, q_rows, h["key_len"], layers=[layer])
    torch.cuda.synchronize()
    x = dev(x0)
    dp = {k: dev(v) for k, v in p.items()}
    c.cross_block(layer, x, dp["WQ"], dp["WO"], d["key_len"], ln_gamma=dp["gamma"], ln_beta=dp["beta"],
                  bQ=dp["bQ"], bO=dp["bO"])
    ref = O.cross_block(x0, layer, host(c.Kc), host(c.Vc), h["key_len"], p["WQ"], p["WO"], p["gamma"], p["beta"],
                        1e-5, p["bQ"], p["bO"])
    assert (pos[:, layer] >= 0).any()
    got = host(x)
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= {"f32": 2e-4, "bf16": 2e-2}[cache_dtype]


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_self_attention_step_new_key_dominates(cache_dtype):
    """At two steps the appended key is planted along that step's query, so the
    step's output is the appended V row, which the kernel takes from its inputs
    rather than from the cache row it streams; later steps see that key at large
    scores of either sign."""
    B, L, H, T, S = 4, 2, 3, 448, 40
    c = cxa.CrossAttentionCache(B, T, L, H, 64, cache_dtype)
    rng = np.random.default_rng(956)
    Qs = rng.standard_normal((S, B, L, H, 64)).astype(np.float32)
    Ks = rng.standard_normal((S, B, L, H, 64)).astype(np.float32)
    Vs = rng.standard_normal((S, B, L, H, 64)).astype(np.float32)
    for s in (0, 23):
        q = Qs[s].astype(np.float64)
        alpha = SPIKE_SCORE / (0.125 * np.einsum("blhc,blhc->blh", q, q))
        Ks[s] = (alpha[..., None] * q).astype(np.float32)
    if cache_dtype == "bf16":
        Ks, Vs = W.bf16_round(Ks), W.bf16_round(Vs)
    outs = [torch.empty((B, L, H, 64), device="cuda") for _ in range(S)]
    Qd, Kd, Vd = [dev(x) for x in Qs], [dev(x) for x in Ks], [dev(x) for x in Vs]
    pos = [dev(np.full(B, s, np.int32), torch.int32) for s in range(S)]
    torch.cuda.synchronize()
    for s in range(S):
        c.self_attention_step(pos[s], Qd[s], Kd[s], Vd[s], out=outs[s])
    torch.cuda.synchronize()
    got = np.stack([host(o) for o in outs])
    assert np.isfinite(got).all()
    for s in (0, 23):
        assert np.abs(got[s] - Vs[s]).max() <= TOL[cache_dtype]
    for b in range(B):
        for l in range(L):
            for hh in range(H):
                ref = O.self_attention_steps(Qs[:, b, l, hh], Ks[:, b, l, hh], Vs[:, b, l, hh])
                assert np.abs(got[:, b, l, hh] - ref).max() <= TOL[cache_dtype]
