"""cxa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (a host whose device memory all belongs to its own pool
allocator, or a serving loop that must not pay for a fresh cudaMalloc). It
runs the decode kernel with its scratch in libcxa's fixed device array.

Checked here through the C ABI: two calls in a row give the same output as
cxa_decode with a caller-owned workspace; calls that alternate between two
caches of different shape on one stream (so the shared array's counters and
partials are laid out differently from one call to the next) stay exact; a
call after a reported kernel timeout (which re-clears the array) stays exact;
and geometry whose scratch exceeds the fixed maximum is refused without
launching anything. This file is collected
last so that a failure here cannot hide the other tests' results.
"""
import numpy as np
import pytest
import torch

from _gpu_common import (DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, cache_for, decode_policy, dev, host,
                         inputs_on_device)
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W
from oracle import cross_attention as O

pytestmark = pytest.mark.gpu

# Short streams take the cluster-per-row decode, which needs no scratch at all; the
# tests below run the persistent stream kernel, whose split rows use the fixed array.


@pytest.mark.parametrize("shape", ["stream", "auto"])
def test_noalloc_decode_matches_decode_on_two_calls(cxa_lib, shape):
    """Two calls in a row equal cxa_decode (caller-owned workspace) and the oracle."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = W.custom("noalloc", B=4, T=700, d=256, L=2, H=4, ragged=True, index=930)
    assert cxa.cxa_decode_workspace_bytes(w.B, w.T, w.L, w.H) <= cxa.CXA_NOALLOC_SCRATCH_BYTES
    d, h = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    stream = torch.cuda.current_stream()
    Kg, Vg = host(c.Kc), host(c.Vc)
    with decode_policy(shape):
        for step in range(2):
            Qh = W.make_Q(w, step)
            Q = dev(Qh)
            ref = torch.empty_like(Q)
            rc = cxa.cxa_decode(c.handle, Q, d["key_len"], ref, 0.0, c.decode_ws, c.decode_ws_bytes, stream)
            assert rc == cxa.CXA_OK
            got = torch.full_like(Q, float("nan"))
            rc = cxa.cxa_decode_noalloc(c.handle, Q, d["key_len"], got, 0.0, stream)
            assert rc == cxa.CXA_OK, cxa.cxa_last_error_message()
            torch.cuda.synchronize()
            err = (got - ref).abs().max().item()
            assert np.isfinite(err) and err <= DECODE_F32_MAX_ABS, err
            assert np.abs(host(got) - O.decode(Qh, Kg, Vg, h["key_len"])).max() <= DECODE_F32_MAX_ABS
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def test_noalloc_alternating_geometries_on_one_stream(cxa_lib):
    """Two caches of different B, L, H (and cache dtype) take turns in the one
    array without a sync between calls (so its counters and partials are laid out
    differently from one call to the next); each output equals cxa_decode's."""
    w1 = W.custom("na1", B=3, T=900, d=384, L=2, H=6, ragged=True, index=931)
    w2 = W.custom("na2", B=5, T=333, d=128, L=3, H=2, ragged=True, index=932)
    caches = []
    for w, cdt in ((w1, "f32"), (w2, "bf16")):
        d, _ = inputs_on_device(w)
        c = cache_for(w, cdt)
        c.populate(d["E"], d["WK"], d["WV"], d["bV"])
        caches.append((w, c, d))
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    got, ref = [], []
    with decode_policy("stream"):
        for step in range(4):
            for (w, c, d) in caches:
                Q = dev(W.make_Q(w, step))
                r = torch.empty_like(Q)
                rc = cxa.cxa_decode(c.handle, Q, d["key_len"], r, 0.0, c.decode_ws, c.decode_ws_bytes, stream)
                assert rc == cxa.CXA_OK
                g = torch.full_like(Q, float("nan"))
                rc = cxa.cxa_decode_noalloc(c.handle, Q, d["key_len"], g, 0.0, stream)
                assert rc == cxa.CXA_OK, cxa.cxa_last_error_message()
                got.append(g)
                ref.append(r)
        torch.cuda.synchronize()
    tol = [DECODE_F32_MAX_ABS, DECODE_BF16_MAX_ABS] * 4
    for g, r, t in zip(got, ref, tol):
        err = (g - r).abs().max().item()
        assert np.isfinite(err) and err <= t, err
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def test_noalloc_after_a_reported_timeout(cxa_lib):
    """A bounded wait that runs out (the library's self-test, which faults
    nothing) is reported by cxa_device_status; the next call clears the array
    again and still matches cxa_decode."""
    w = W.custom("na3", B=2, T=1500, d=256, L=2, H=4, ragged=True, index=933)
    d, _ = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    assert cxa.cxa_selftest_wait_timeout(2000) == cxa.CXA_OK
    assert cxa.cxa_device_status(1) == cxa.CXA_ETIMEOUT
    Q = dev(W.make_Q(w, 0))
    with decode_policy("stream"):
        ref = c.decode(Q, d["key_len"]).clone()
        got = torch.full_like(Q, float("nan"))
        rc = cxa.cxa_decode_noalloc(c.handle, Q, d["key_len"], got, 0.0)
        assert rc == cxa.CXA_OK, cxa.cxa_last_error_message()
        torch.cuda.synchronize()
    assert (got - ref).abs().max().item() <= DECODE_F32_MAX_ABS
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
