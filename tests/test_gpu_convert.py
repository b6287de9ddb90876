"""The fp32 -> bf16 conversion pass (cxa_convert_bf16) against the oracle's
round_bf16, bit for bit: random bit patterns (every exponent, subnormals,
huge values that round to infinity), exact ties in both directions, infinities
and NaNs, ragged lengths around the 8-value groups, an empty call, and a length
that spans more than one grid stride."""
import numpy as np
import pytest
import torch

from encoder_decoder_speech_gb300 import cxa
from oracle import cross_attention as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _bits_gpu(x: np.ndarray) -> np.ndarray:
    src = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    dst = torch.full((x.size,), -1, dtype=torch.int16, device="cuda")
    assert cxa.cxa_convert_bf16(src, dst, x.size, None) == cxa.CXA_OK, cxa.cxa_last_error_message()
    torch.cuda.synchronize()
    return dst.cpu().numpy().view(np.uint16)


def _bits_oracle(x: np.ndarray) -> np.ndarray:
    return (O.round_bf16(x).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _compare(x):
    got, want = _bits_gpu(x), _bits_oracle(x)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan]), np.flatnonzero(got[~nan] != want[~nan])[:8]
    g = got[nan]
    assert ((g & 0x7F80) == 0x7F80).all() and ((g & 0x7F) != 0).all()     # NaN stays NaN


@pytest.mark.parametrize("n", [1, 7, 8, 9, 15, 16, 17, 1000, 4099])
def test_random_patterns_ragged_lengths(n):
    rng = np.random.default_rng(1000 + n)
    x = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    _compare(x)


def test_ties_specials_and_subnormals():
    base = np.array([1.0, -1.0, 3.0, 1e-3, 1e30, 2.0 ** -130], dtype=np.float32).view(np.uint32)
    pats = []
    for b in base:
        hi = b & np.uint32(0xFFFF0000)
        pats += [hi | np.uint32(0x8000), hi | np.uint32(0x4000),
                 hi | np.uint32(0x7FFF), hi | np.uint32(0x8001), (hi + np.uint32(0x10000)) | np.uint32(0x8000)]
    x = np.array(pats, dtype=np.uint32).view(np.float32)
    special = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, np.finfo(np.float32).max, -np.finfo(np.float32).max,
                        np.finfo(np.float32).tiny, 1e-45, -1e-45, 3.389e38, 3.3895e38, 3.3903e38],
                       dtype=np.float32)
    _compare(np.concatenate([x, special]))


def test_large_length_and_empty_call():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(152 * 8 * 256 * 8 * 3 + 5) * 10.0).astype(np.float32)
    _compare(x)
    src = torch.zeros(16, device="cuda")
    dst = torch.zeros(16, dtype=torch.int16, device="cuda")
    before = cxa.cxa_launch_count()
    assert cxa.cxa_convert_bf16(src, dst, 0, None) == cxa.CXA_OK
    assert cxa.cxa_launch_count() == before


def test_misaligned_or_overlapping_buffers_are_refused():
    src = torch.zeros(64, device="cuda")
    dst = torch.zeros(64, dtype=torch.int16, device="cuda")
    assert cxa.cxa_convert_bf16(src.data_ptr() + 4, dst, 8, None) == cxa.CXA_EINVAL
    assert cxa.cxa_convert_bf16(src, dst.data_ptr() + 2, 8, None) == cxa.CXA_EINVAL
    assert cxa.cxa_convert_bf16(src, src, 8, None) == cxa.CXA_EINVAL
