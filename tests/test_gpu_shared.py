"""Parity of cxa_decode_shared (nq hypotheses per slot attending the slot's one
cache) with the oracle's decode_shared, kernel-isolated: the oracle decodes the
very cache the GPU holds."""
import numpy as np
import pytest
import torch

from _gpu_common import DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, cache_for, dev, host, inputs_on_device
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


def _queries(w, nq, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((w.B, nq, w.L, w.H, 64)).astype(np.float32)


@pytest.mark.parametrize("cache_dtype,nq", [(c, n) for c in ("f32", "bf16") for n in (1, 2, 3, 4, 5, 6, 7, 8)]
                         + [("bf16", n) for n in (9, 12, 16)])
def test_shared_decode_matches_oracle(nq, cache_dtype):
    w = W.custom("shared", B=4, T=700, d=256, L=2, H=4, ragged=True, index=940)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    kl = h["key_len"].copy()
    kl[2] = 0                                   # an empty slot gets zeros
    Q = _queries(w, nq, nq)
    out = host(c.decode_shared(dev(Q), dev(kl, torch.int32)))
    ref = O.decode_shared(Q, host(c.Kc), host(c.Vc), kl)
    assert np.abs(out - ref).max() <= TOL[cache_dtype]
    assert np.all(out[2] == 0.0)


def test_shared_decode_with_one_query_is_decode():
    w = W.custom("shared1", B=3, T=500, d=128, L=3, H=2, ragged=True, index=941)
    d, _ = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Q = dev(W.make_Q(w, 0))
    a = c.decode(Q, d["key_len"])
    b = c.decode_shared(Q[:, None].contiguous(), d["key_len"])[:, 0]
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_shared_decode_back_to_back_and_invalid_nq():
    w = W.custom("shared_b2b", B=2, T=1300, d=512, L=2, H=8, ragged=True, index=942)
    d, h = inputs_on_device(w)
    c = cache_for(w, "bf16")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Qs = [_queries(w, 5, 50 + s) for s in range(6)]
    outs = [c.decode_shared(dev(q), d["key_len"]) for q in Qs]
    torch.cuda.synchronize()
    K, V = host(c.Kc), host(c.Vc)
    for q, o in zip(Qs, outs):
        assert np.abs(host(o) - O.decode_shared(q, K, V, h["key_len"])).max() <= DECODE_BF16_MAX_ABS
    Q17 = dev(_queries(w, 17, 1))
    out = torch.empty_like(Q17)
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device="cuda")
    assert cxa.cxa_decode_shared(c.handle, 17, Q17, d["key_len"], out, 0.0, ws, ws.numel()) == cxa.CXA_EINVAL
    assert cxa.cxa_decode_shared(c.handle, 0, Q17, d["key_len"], out, 0.0, ws, ws.numel()) == cxa.CXA_EINVAL
    c32 = cache_for(w, "f32")
    c32.populate(d["E"], d["WK"], d["WV"], d["bV"])
    assert cxa.cxa_decode_shared(c32.handle, 9, Q17, d["key_len"], out, 0.0, ws, ws.numel()) == cxa.CXA_EINVAL


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_batched_base_beam5(cache_dtype):
    """Batched Whisper-Base with 5 hypotheses per memory (a beam of 5), all rows."""
    w = W.WORKLOADS["batched_base"]
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Q = _queries(w, 5, 7)
    out = host(c.decode_shared(dev(Q), d["key_len"]))
    ref = O.decode_shared(Q, host(c.Kc), host(c.Vc), h["key_len"])
    assert np.abs(out - ref).max() <= TOL[cache_dtype]


@pytest.mark.parametrize("nq", [3, 8, 16])
def test_shared_decode_growing_scores_move_the_reference(nq):
    """Key rows scaled up along t make later chunks' scores pass the running max
    by far more than the 2^8 margin inside row segments, so the tensor-core
    decode rescales its O accumulator in tensor memory; the result must still
    match the oracle."""
    w = W.custom("shared_grow", B=8, T=1500, d=512, L=2, H=8, ragged=True, index=943)
    d, h = inputs_on_device(w)
    c = cache_for(w, "bf16")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    ramp = 1.0 + torch.arange(w.T, device="cuda", dtype=torch.float32) / 48.0
    c.Kc.mul_(ramp.to(c.Kc.dtype)[:, None])
    Q = (3.0 * _queries(w, nq, 60 + nq)).astype(np.float32)
    K, V = host(c.Kc), host(c.Vc)
    # precondition: chunk maxima (log2 units) jump past the running max by > 8
    s = np.einsum("bqlhc,blhtc->bqlht", Q.astype(np.float64), K) * (64 ** -0.5) / np.log(2.0)
    jumps = 0
    for b in range(w.B):
        n = int(h["key_len"][b])
        cm = [s[b, ..., t0:min(n, t0 + 128)].max(-1) for t0 in range(0, n, 128)]
        run = cm[0]
        for m in cm[1:]:
            jumps += int(np.sum(m > run + 8.0))
            run = np.maximum(run, m)
    assert jumps > 100
    out = host(c.decode_shared(dev(Q), d["key_len"]))
    ref = O.decode_shared(Q, K, V, h["key_len"])
    assert np.abs(out - ref).max() <= DECODE_BF16_MAX_ABS


@pytest.mark.parametrize("nq", [3, 8, 16])
def test_shared_decode_tensor_core_key_length_edges(nq):
    """Key lengths at and around the 32-key TMA boxes and 128-key chunks (1, 2, 31,
    32, 33, 127, 128, 129, T) on a bf16 cache: tail rows of a chunk are stale data
    that must not reach the output."""
    w = W.custom("shared_edges", B=9, T=333, d=256, L=2, H=4, ragged=False, index=944)
    d, h = inputs_on_device(w)
    c = cache_for(w, "bf16")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    kl = np.array([1, 2, 31, 32, 33, 127, 128, 129, 333], dtype=np.int32)
    Q = _queries(w, nq, 70 + nq)
    out = host(c.decode_shared(dev(Q), dev(kl, torch.int32)))
    ref = O.decode_shared(Q, host(c.Kc), host(c.Vc), kl)
    assert np.abs(out - ref).max() <= DECODE_BF16_MAX_ABS


@pytest.mark.parametrize("nq", [3, 4, 5, 6, 8])
def test_shared_decode_fp32_key_length_edges(nq):
    """fp32 cache, several queries (one key per lane in each 32-key half of a 64-key
    chunk): key lengths at and around the halves and chunks (1, 2, 31, 32, 33, 63,
    64, 65, T). Keys past the length are stale rows that must not reach the output."""
    w = W.custom("shared_edges32", B=9, T=333, d=256, L=2, H=4, ragged=False, index=946)
    d, h = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    kl = np.array([1, 2, 31, 32, 33, 63, 64, 65, 333], dtype=np.int32)
    Q = _queries(w, nq, 90 + nq)
    out = host(c.decode_shared(dev(Q), dev(kl, torch.int32)))
    ref = O.decode_shared(Q, host(c.Kc), host(c.Vc), kl)
    assert np.abs(out - ref).max() <= DECODE_F32_MAX_ABS


def test_shared_decode_clamps_key_lengths():
    """key_len outside [0, T] is clamped (negative -> no key -> zeros; > T -> T)."""
    w = W.custom("shared_clamp", B=4, T=200, d=256, L=2, H=4, ragged=False, index=945)
    d, h = inputs_on_device(w)
    c = cache_for(w, "bf16")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    kl = np.array([-5, 0, 200, 100000], dtype=np.int32)
    Q = _queries(w, 6, 80)
    out = host(c.decode_shared(dev(Q), dev(kl, torch.int32)))
    ref = O.decode_shared(Q, host(c.Kc), host(c.Vc), np.clip(kl, 0, w.T))
    assert np.abs(out - ref).max() <= DECODE_BF16_MAX_ABS
    assert np.all(out[0] == 0.0) and np.all(out[1] == 0.0)


@pytest.mark.parametrize("nq", [2, 4, 8, 16])
@pytest.mark.parametrize("geom", ["one_long_memory", "mixed_lengths"])
def test_shared_decode_rows_cut_many_times(nq, geom):
    """Rows far longer than a CTA's share of the chunks, so that range boundaries cut
    each row tens of times (about 76 segments per row for one 32768-key memory of
    4 rows): every cut row is merged once, from all of its segments in order
    (in the kernel for up to four queries, by the merge kernel for more)."""
    if geom == "one_long_memory":
        w = W.custom("shared_cut", B=1, T=32768, d=128, L=2, H=2, ragged=False, index=947)
        kl = np.array([32763], dtype=np.int32)
    else:
        w = W.custom("shared_cut_mixed", B=3, T=4096, d=128, L=2, H=2, ragged=False, index=948)
        kl = np.array([4096, 1, 2500], dtype=np.int32)
    d, h = inputs_on_device(w)
    c = cache_for(w, "bf16")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Q = _queries(w, nq, 110 + nq)
    kld = dev(kl, torch.int32)
    outs = [c.decode_shared(dev(Q), kld) for _ in range(2)]
    out = host(outs[1])
    ref = O.decode_shared(Q, host(c.Kc), host(c.Vc), kl)
    assert np.abs(out - ref).max() <= DECODE_BF16_MAX_ABS
    assert torch.equal(outs[0], outs[1])
