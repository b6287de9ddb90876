"""cxa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (a host whose device memory all belongs to its own pool
allocator, or a serving loop that must not pay for a fresh cudaMalloc). It
runs the decode kernel with its scratch in libcxa's fixed device array.

Checked here through the C ABI: two calls in a row give the same output as
cxa_decode with a caller-owned workspace, and geometry whose scratch exceeds
the fixed maximum is refused without launching anything. This file is collected
last so that a failure here cannot hide the other tests' results.
"""
import numpy as np
import pytest
import torch

from _gpu_common import DECODE_F32_MAX_ABS, cache_for, dev, inputs_on_device
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_decode_on_two_calls(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = W.custom("noalloc", B=4, T=700, d=256, L=2, H=4, ragged=True, index=930)
    assert cxa.cxa_decode_workspace_bytes(w.B, w.T, w.L, w.H) <= cxa.CXA_NOALLOC_SCRATCH_BYTES
    d, _ = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    stream = torch.cuda.current_stream()
    for step in range(2):
        Q = dev(W.make_Q(w, step))
        ref = torch.empty_like(Q)
        assert cxa.cxa_decode(c.handle, Q, d["key_len"], ref, 0.0, c.decode_ws, c.decode_ws_bytes, stream) == cxa.CXA_OK
        got = torch.full_like(Q, float("nan"))
        rc = cxa.cxa_decode_noalloc(c.handle, Q, d["key_len"], got, 0.0, stream)
        assert rc == cxa.CXA_OK, cxa.cxa_last_error_message()
        torch.cuda.synchronize()
        err = (got - ref).abs().max().item()
        assert np.isfinite(err) and err <= DECODE_F32_MAX_ABS, err
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def test_noalloc_refuses_geometry_beyond_its_scratch(cxa_lib):
    # batched-Base-sized rows at T = 32768 need far more than the fixed scratch
    B, T, L, H = 16, 32768, 6, 8
    assert cxa.cxa_decode_workspace_bytes(B, T, L, H) > cxa.CXA_NOALLOC_SCRATCH_BYTES
    fake = 0x7f0000000000
    rc, h = cxa.cxa_cache_create(fake, fake + (1 << 36), B, T, L, H, 64, cxa.CXA_F32)
    assert rc == cxa.CXA_OK
    before = cxa.cxa_launch_count()
    rc = cxa.cxa_decode_noalloc(h, fake, fake, fake + 4096, 0.0, 0)
    assert rc == cxa.CXA_EINVAL
    assert "fixed maximum" in cxa.cxa_last_error_message()
    assert cxa.cxa_launch_count() == before
    cxa.cxa_cache_destroy(h)
