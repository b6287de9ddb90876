"""Failure detection on the GPU without a fault: a kernel's bounded wait on a
barrier that nothing completes gives up after a short limit, sets the device
status word and returns; the host reads CXA_ETIMEOUT, clears it, and the context
goes on working (a decode right after still matches the oracle)."""
import time

import numpy as np
import pytest
import torch

from _gpu_common import DECODE_F32_MAX_ABS, cache_for, dev, host, inputs_on_device
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W
from oracle import cross_attention as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.synchronize()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def test_bounded_wait_expires_and_is_reported():
    assert cxa.cxa_device_status(1) == cxa.CXA_OK          # start clean
    t0 = time.perf_counter()
    assert cxa.cxa_selftest_wait_timeout(20000) == cxa.CXA_OK   # a 20 ms limit
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 0.015 <= waited < 5.0                           # it waited, and it came back
    assert cxa.cxa_device_status(1) == cxa.CXA_ETIMEOUT    # reported, and cleared
    assert cxa.cxa_device_status(0) == cxa.CXA_OK
    # the context is still usable
    w = W.custom("after_timeout", B=2, T=100, d=128, L=1, H=2, index=990)
    d, h = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    Q = W.make_Q(w, 0)
    out = host(c.decode(dev(Q), d["key_len"]))
    ref = O.decode(Q, host(c.Kc), host(c.Vc), h["key_len"])
    assert np.abs(out - ref).max() <= DECODE_F32_MAX_ABS
    assert cxa.cxa_device_status(0) == cxa.CXA_OK


def test_selftest_rejects_bad_limits():
    assert cxa.cxa_selftest_wait_timeout(0) == cxa.CXA_EINVAL
    assert cxa.cxa_selftest_wait_timeout(1000001) == cxa.CXA_EINVAL
