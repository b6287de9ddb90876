"""Parity of the per-layer entry points with the oracle: cxa_decode_layers (a
layer range of the cache) and cxa_cross_block (LayerNorm -> Q projection ->
attention over one layer -> out projection + residual), both kernel-isolated:
the oracle works on the very cache the GPU holds.

Block tolerance: everything runs in fp32; beyond the decode bar (1e-4 on an fp32
cache, 1e-2 on a bf16 cache) the two d x d projections add fp32 rounding of
d-term sums, so the block is held to 2e-4 (fp32 cache) and 2e-2 (bf16 cache)."""
import numpy as np
import pytest
import torch

from _gpu_common import DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, cache_for, dev, host, inputs_on_device
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W
from oracle import cross_attention as O

pytestmark = pytest.mark.gpu

DEC_TOL = {"f32": DECODE_F32_MAX_ABS, "bf16": DECODE_BF16_MAX_ABS}
BLOCK_TOL = {"f32": 2e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.synchronize()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def _rand(shape, seed, std=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * std).astype(np.float32)


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("l0,nl", [(0, 4), (2, 1), (1, 3), (3, 1)])
def test_decode_layers(l0, nl, cache_dtype):
    w = W.custom("layers", B=3, T=600, d=256, L=4, H=4, ragged=True, index=950)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Q = _rand((w.B, nl, w.H, 64), 10 * l0 + nl)
    out = host(c.decode_layers(l0, dev(Q), d["key_len"]))
    ref = O.decode_layers(Q, host(c.Kc), host(c.Vc), h["key_len"], l0)
    assert np.abs(out - ref).max() <= DEC_TOL[cache_dtype]


def _block_params(d, seed, with_affine=True):
    p = {"WQ": _rand((d, d), seed, d ** -0.5), "WO": _rand((d, d), seed + 1, d ** -0.5)}
    if with_affine:
        p.update(gamma=1.0 + _rand((d,), seed + 2, 0.1), beta=_rand((d,), seed + 3, 0.1),
                 bQ=_rand((d,), seed + 4, 0.02), bO=_rand((d,), seed + 5, 0.02))
    return p


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_affine", [True, False])
def test_cross_block(cache_dtype, with_affine):
    w = W.custom("block", B=5, T=400, d=256, L=3, H=4, ragged=True, index=951)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    p = _block_params(w.d, 60, with_affine)
    x0 = _rand((w.B, w.d), 61)
    x = dev(x0)
    dp = {k: dev(v) for k, v in p.items()}
    c.cross_block(1, x, dp["WQ"], dp["WO"], d["key_len"], ln_gamma=dp.get("gamma"), ln_beta=dp.get("beta"),
                  bQ=dp.get("bQ"), bO=dp.get("bO"))
    ref = O.cross_block(x0, 1, host(c.Kc), host(c.Vc), h["key_len"], p["WQ"], p["WO"], p.get("gamma"),
                        p.get("beta"), 1e-5, p.get("bQ"), p.get("bO"))
    assert np.abs(host(x) - ref).max() <= BLOCK_TOL[cache_dtype]


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("H", [1, 6, 10])
def test_cross_block_head_counts(cache_dtype, H):
    """Up to 8 heads the block runs as one kernel (a cluster of H CTAs per slot),
    beyond that as three; an empty slot (key_len 0) gets x += bO only."""
    w = W.custom("blockH%d" % H, B=3, T=300, d=64 * H, L=2, H=H, ragged=True, index=960 + H)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    p = _block_params(w.d, 62 + H)
    kl = h["key_len"].copy()
    kl[1] = 0
    x0 = _rand((w.B, w.d), 63 + H)
    x = dev(x0)
    dp = {k: dev(v) for k, v in p.items()}
    c.cross_block(1, x, dp["WQ"], dp["WO"], dev(kl, torch.int32), ln_gamma=dp["gamma"], ln_beta=dp["beta"],
                  bQ=dp["bQ"], bO=dp["bO"])
    ref = O.cross_block(x0, 1, host(c.Kc), host(c.Vc), kl, p["WQ"], p["WO"], p["gamma"], p["beta"], 1e-5,
                        p["bQ"], p["bO"])
    assert np.abs(host(x) - ref).max() <= BLOCK_TOL[cache_dtype]


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_interleaved_layers_batched_base(cache_dtype):
    """Batched Whisper-Base: the six layers' blocks applied in turn to the residual
    stream, as a decoder step does, launched back to back without syncs."""
    w = W.WORKLOADS["batched_base"]
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    params = [_block_params(w.d, 70 + 10 * l) for l in range(w.L)]
    dparams = [{k: dev(v) for k, v in p.items()} for p in params]
    x0 = _rand((w.B, w.d), 69)
    x = dev(x0)
    torch.cuda.synchronize()
    for l in range(w.L):
        dp = dparams[l]
        c.cross_block(l, x, dp["WQ"], dp["WO"], d["key_len"], ln_gamma=dp["gamma"], ln_beta=dp["beta"],
                      bQ=dp["bQ"], bO=dp["bO"])
    got = host(x)
    K, V = host(c.Kc), host(c.Vc)
    ref = x0.astype(np.float64)
    for l in range(w.L):
        p = params[l]
        ref = O.cross_block(ref, l, K, V, h["key_len"], p["WQ"], p["WO"], p["gamma"], p["beta"], 1e-5, p["bQ"],
                            p["bO"])
    assert np.abs(got - ref).max() <= BLOCK_TOL[cache_dtype]


def test_block_argument_checks():
    w = W.custom("blockarg", B=2, T=100, d=128, L=2, H=2, index=952)
    d, _ = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    x = torch.zeros((w.B, w.d), device="cuda")
    Wm = torch.zeros((w.d, w.d), device="cuda")
    ws = torch.zeros(cxa.cxa_cross_block_workspace_bytes(w.B, w.T, w.L, w.H), dtype=torch.uint8, device="cuda")
    args = lambda layer: (c.handle, layer, x, None, None, 1e-5, Wm, None, Wm, None, d["key_len"], 0.0, ws, ws.numel())
    assert cxa.cxa_cross_block(*args(2)) == cxa.CXA_EINVAL
    assert cxa.cxa_cross_block(*args(-1)) == cxa.CXA_EINVAL
    c.invalidate(0)
    assert cxa.cxa_cross_block(*args(0)) == cxa.CXA_ENOTREADY


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_cross_block_clamps_key_lengths(cache_dtype):
    """key_len outside [0, T]: negative attends nothing (x += bO), beyond T attends all T."""
    w = W.custom("blockclamp", B=3, T=250, d=256, L=2, H=4, ragged=False, index=966)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    p = _block_params(w.d, 67)
    kl = np.array([-3, 400, 120], dtype=np.int32)
    x0 = _rand((w.B, w.d), 68)
    x = dev(x0)
    dp = {k: dev(v) for k, v in p.items()}
    c.cross_block(0, x, dp["WQ"], dp["WO"], dev(kl, torch.int32), ln_gamma=dp["gamma"], ln_beta=dp["beta"],
                  bQ=dp["bQ"], bO=dp["bO"])
    ref = O.cross_block(x0, 0, host(c.Kc), host(c.Vc), np.clip(kl, 0, w.T), p["WQ"], p["WO"], p["gamma"],
                        p["beta"], 1e-5, p["bQ"], p["bO"])
    assert np.abs(host(x) - ref).max() <= BLOCK_TOL[cache_dtype]


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_cross_block_key_lengths_around_chunks(cache_dtype):
    """Rows ending just before, on and after the ring's chunk boundaries (24 fp32 /
    48 bf16 keys per stage; 96 and 192 are whole chunks of both) and around the ring's
    depth (16 stages: 384 fp32 keys)."""
    kls = [1, 95, 96, 97, 191, 192, 193, 383, 384, 385, 700]
    w = W.custom("blockchunks", B=len(kls), T=700, d=256, L=2, H=4, ragged=False, index=967)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    p = _block_params(w.d, 69)
    kl = np.array(kls, dtype=np.int32)
    x0 = _rand((w.B, w.d), 70)
    x = dev(x0)
    dp = {k: dev(v) for k, v in p.items()}
    c.cross_block(1, x, dp["WQ"], dp["WO"], dev(kl, torch.int32), ln_gamma=dp["gamma"], ln_beta=dp["beta"],
                  bQ=dp["bQ"], bO=dp["bO"])
    ref = O.cross_block(x0, 1, host(c.Kc), host(c.Vc), kl, p["WQ"], p["WO"], p["gamma"], p["beta"], 1e-5,
                        p["bQ"], p["bO"])
    assert np.abs(host(x) - ref).max() <= BLOCK_TOL[cache_dtype]


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [16, 17, 19, 21])
def test_cross_block_slot_counts(cache_dtype, B):
    """Eight heads and more slots than the head clusters that fit at once: the
    block clusters along the slots (4 or 2 per cluster, the grid padded to whole
    clusters) or not at all, whichever fits; every form must agree with the oracle."""
    w = W.custom("blockB%d" % B, B=B, T=300, d=512, L=2, H=8, ragged=True, index=970 + B)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    p = _block_params(w.d, 71 + B)
    kl = h["key_len"].copy()
    kl[B // 2] = 0
    x0 = _rand((w.B, w.d), 72 + B)
    x = dev(x0)
    dp = {k: dev(v) for k, v in p.items()}
    c.cross_block(1, x, dp["WQ"], dp["WO"], dev(kl, torch.int32), ln_gamma=dp["gamma"], ln_beta=dp["beta"],
                  bQ=dp["bQ"], bO=dp["bO"])
    ref = O.cross_block(x0, 1, host(c.Kc), host(c.Vc), kl, p["WQ"], p["WO"], p["gamma"], p["beta"], 1e-5,
                        p["bQ"], p["bO"])
    assert np.abs(host(x) - ref).max() <= BLOCK_TOL[cache_dtype]
