"""Alignment-head cross-attention weights on the GPU against the oracle
(kernel-isolated: the oracle reads the GPU's own cache): rows of selected
(layer, head) pairs, their mean over heads, sums of 1 over valid keys, zeros
beyond key_len, and weights x V equal to the decode output of the same head.
Probabilities are fp32 softmax values (<= 1), held to 1e-5 absolute."""
import numpy as np
import pytest
import torch

from _gpu_common import DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, cache_for, dev, host, inputs_on_device
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W
from oracle import cross_attention as O

pytestmark = pytest.mark.gpu
WEIGHT_MAX_ABS = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.synchronize()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 17, 1500])
def test_alignment_weights(cache_dtype, T):
    w = W.custom("align", B=4, T=T, d=256, L=3, H=4, ragged=True, index=960)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    kl = h["key_len"].copy()
    kl[3] = 0
    heads = [(0, 0), (2, 3), (1, 1), (2, 0), (0, 3)]
    Q = W.make_Q(w, 3)
    wt, mean = c.alignment_weights(dev(Q), dev(kl, torch.int32), heads)
    out = host(c.decode(dev(Q), dev(kl, torch.int32)))
    wt, mean = host(wt), host(mean)
    K, V = host(c.Kc), host(c.Vc)
    ref_w, ref_m = O.attention_weights(Q, K, kl, heads)
    assert np.abs(wt - ref_w).max() <= WEIGHT_MAX_ABS
    assert np.abs(mean - ref_m).max() <= WEIGHT_MAX_ABS
    for b in range(w.B):
        for k, (l, hh) in enumerate(heads):
            n = min(max(int(kl[b]), 0), T)
            assert np.all(wt[b, k, n:] == 0.0)
            assert abs(wt[b, k].sum() - (1.0 if n else 0.0)) <= 1e-5
            tol = DECODE_F32_MAX_ABS if cache_dtype == "f32" else DECODE_BF16_MAX_ABS
            assert np.abs(wt[b, k] @ V[b, l, hh] - out[b, l, hh]).max() <= tol


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_alignment_sixteen_slots_narrow_ring(cache_dtype):
    """Sixteen slots and six heads (the batched Whisper-Base shape of a call): the
    launch takes the 8 x 8 KB ring there, whose clusters can be 16 CTAs, against the
    oracle, with ragged, empty and full key lengths."""
    w = W.custom("align16", B=16, T=1500, d=512, L=6, H=8, ragged=True, index=964)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    kl = h["key_len"].copy()
    kl[5], kl[11] = 0, w.T
    heads = [(3, 1), (4, 2), (4, 6), (5, 0), (5, 3), (5, 7)]
    Q = W.make_Q(w, 5)
    wt, mean = c.alignment_weights(dev(Q), dev(kl, torch.int32), heads)
    wt, mean = host(wt), host(mean)
    ref_w, ref_m = O.attention_weights(Q, host(c.Kc), kl, heads)
    assert np.abs(wt - ref_w).max() <= WEIGHT_MAX_ABS
    assert np.abs(mean - ref_m).max() <= WEIGHT_MAX_ABS
    assert np.all(wt[5] == 0.0) and np.all(mean[5] == 0.0)


def test_alignment_weights_large_dims():
    """Whisper-large dims (32 layers, 20 heads, bf16 cache), a spread of heads."""
    w = W.WORKLOADS["large"]
    d, h = inputs_on_device(w)
    c = cache_for(w, "bf16")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    heads = [(l, (7 * l) % w.H) for l in range(16, 32, 2)]
    Q = W.make_Q(w, 9)
    wt, mean = c.alignment_weights(dev(Q), d["key_len"], heads)
    ref_w, ref_m = O.attention_weights(Q, host(c.Kc), h["key_len"], heads)
    assert np.abs(host(wt) - ref_w).max() <= WEIGHT_MAX_ABS
    assert np.abs(host(mean) - ref_m).max() <= WEIGHT_MAX_ABS


def test_alignment_argument_checks():
    w = W.custom("align_args", B=2, T=50, d=128, L=2, H=2, index=961)
    d, _ = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Q = dev(W.make_Q(w, 0))
    wt = torch.empty((w.B, 1, w.T), device="cuda")
    assert cxa.cxa_alignment_weights(c.handle, Q, d["key_len"], [(2, 0)], wt, None, 0.0) == cxa.CXA_EINVAL
    assert cxa.cxa_alignment_weights(c.handle, Q, d["key_len"], [(0, 2)], wt, None, 0.0) == cxa.CXA_EINVAL
    assert cxa.cxa_alignment_weights(c.handle, Q, d["key_len"], [], wt, None, 0.0) == cxa.CXA_EINVAL


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_alignment_key_lengths_around_cluster_split(cache_dtype):
    """Key lengths shorter than, equal to and just past the per-CTA key ranges of a
    slot's cluster, negative and beyond T; outputs pre-filled with NaN must be
    overwritten everywhere."""
    kls = [1, 7, 8, 9, 15, 16, 17, 31, 33, 129, 300, -4, 5000, 0]
    w = W.custom("align_edges", B=len(kls), T=300, d=256, L=2, H=4, ragged=False, index=962)
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    kl = np.array(kls, dtype=np.int32)
    heads = [(1, 2), (0, 0), (1, 3)]
    Q = W.make_Q(w, 4)
    wt = torch.full((w.B, len(heads), w.T), float("nan"), device="cuda")
    mean = torch.full((w.B, w.T), float("nan"), device="cuda")
    assert cxa.cxa_alignment_weights(c.handle, dev(Q), dev(kl, torch.int32), heads, wt, mean, 0.0) == cxa.CXA_OK
    wt, mean = host(wt), host(mean)
    ref_w, ref_m = O.attention_weights(Q, host(c.Kc), np.clip(kl, 0, w.T), heads)
    assert np.all(np.isfinite(wt)) and np.all(np.isfinite(mean))
    assert np.abs(wt - ref_w).max() <= WEIGHT_MAX_ABS
    assert np.abs(mean - ref_m).max() <= WEIGHT_MAX_ABS


def test_alignment_many_heads_long_rows_no_mean():
    """64 selected heads (the maximum, with repeats) over 8192 keys: several load
    batches per CTA; the mean is not requested."""
    w = W.custom("align_many", B=3, T=8192, d=256, L=4, H=4, ragged=True, index=963)
    d, h = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    heads = [((5 * k) % w.L, (3 * k + 1) % w.H) for k in range(64)]
    Q = W.make_Q(w, 5)
    wt, mean = c.alignment_weights(dev(Q), d["key_len"], heads, with_mean=False)
    assert mean is None
    ref_w, _ = O.attention_weights(Q, host(c.Kc), h["key_len"], heads)
    assert np.abs(host(wt) - ref_w).max() <= WEIGHT_MAX_ABS
