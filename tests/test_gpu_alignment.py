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
