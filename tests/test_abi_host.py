"""Host-side tests of the C ABI: the library builds and loads, exports every symbol
include/cxa.h declares, and validates arguments and ready flags before touching
CUDA. No GPU is needed: every call here fails or returns before any CUDA call,
and the pointers handed over are never dereferenced."""
import ctypes
import os
import re

import pytest

from encoder_decoder_speech_gb300 import cxa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "cxa.h")
FAKE = 0x7f0000000000          # 256-byte aligned, never dereferenced
BIG = 1 << 40


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CXA_API\s+[\w\s\*]+?\b(cxa_\w+)\s*\(", text)))


def test_header_declares_the_documented_calls():
    names = declared_symbols()
    for n in ["cxa_populate", "cxa_decode", "cxa_invalidate", "cxa_cache_create", "cxa_cache_destroy"]:
        assert n in names
    assert set(names) == set(cxa.SIGNATURES)


def test_library_exports_every_declared_symbol(cxa_lib):
    for name in declared_symbols():
        assert hasattr(cxa_lib, name), name
        assert ctypes.cast(getattr(cxa_lib, name), ctypes.c_void_p).value


def make(B=2, T=1500, L=6, H=8, dh=64, dtype=cxa.CXA_F32, Kc=FAKE, Vc=FAKE + (1 << 32)):
    return cxa.cxa_cache_create(Kc, Vc, B, T, L, H, dh, dtype)


def test_create_validates_geometry(cxa_lib):
    rc, h = make()
    assert rc == cxa.CXA_OK and h
    cxa.cxa_cache_destroy(h)
    assert make(T=0)[0] == cxa.CXA_EINVAL          # positive encoder memory length
    assert make(T=-5)[0] == cxa.CXA_EINVAL
    assert make(dh=32)[0] == cxa.CXA_EINVAL        # build specialised to dh = 64
    assert make(B=0)[0] == cxa.CXA_EINVAL
    assert make(dtype=7)[0] == cxa.CXA_EINVAL
    assert make(Kc=0)[0] == cxa.CXA_EINVAL
    assert make(Kc=FAKE + 8)[0] == cxa.CXA_EINVAL  # not 16-byte aligned
    assert "aligned" in cxa.cxa_last_error_message()


def test_workspace_sizes(cxa_lib):
    assert cxa.cxa_populate_workspace_bytes(512, 6, cxa.CXA_F32) == 2 * 6 * 512 * 512 * 4
    assert cxa.cxa_populate_workspace_bytes(1280, 32, cxa.CXA_BF16) == 2 * 32 * 1280 * 1280 * 2
    n = cxa.cxa_decode_workspace_bytes(16, 1500, 6, 8)
    assert n >= 16 * 6 * 8 * 24 * 68 * 4
    assert cxa.cxa_decode_workspace_bytes(16, 1500, 6, 8, 32) == 0


def test_decode_refuses_until_populated(cxa_lib):
    """A never-populated or invalidated cache makes decode return -2 and launch nothing."""
    rc, h = make()
    assert cxa.cxa_is_ready(h, 0) == 0
    before = cxa.cxa_launch_count()
    rc = cxa.cxa_decode(h, FAKE, FAKE, FAKE + 4096, 0.0, FAKE + 8192, BIG, 0)
    assert rc == cxa.CXA_ENOTREADY
    assert "not populated" in cxa.cxa_last_error_message()
    assert cxa.cxa_launch_count() == before
    assert cxa.cxa_strerror(rc).startswith("CXA_ENOTREADY")
    cxa.cxa_cache_destroy(h)


def test_decode_argument_checks(cxa_lib):
    rc, h = make()
    assert cxa.cxa_decode(h, 0, FAKE, FAKE, 0.0, FAKE, BIG, 0) == cxa.CXA_EINVAL
    assert cxa.cxa_decode(h, FAKE + 4, FAKE, FAKE + 4096, 0.0, FAKE, BIG, 0) == cxa.CXA_EINVAL
    assert cxa.cxa_decode(h, FAKE, FAKE, FAKE, 0.0, FAKE, BIG, 0) == cxa.CXA_EINVAL       # out aliases Q
    assert cxa.cxa_decode(h, FAKE, FAKE, FAKE + 4096, 0.0, FAKE, 16, 0) == cxa.CXA_EINVAL  # short workspace
    assert cxa.cxa_decode(h, FAKE, FAKE, FAKE + 4096, float("nan"), FAKE, BIG, 0) == cxa.CXA_EINVAL
    cxa.cxa_cache_destroy(h)


def test_populate_fails_closed_on_geometry(cxa_lib):
    rc, h = make(B=2, T=1500, L=6, H=8)
    args = dict(b0=0, nb=1, E=FAKE, WK=FAKE, WV=FAKE, bV=FAKE, T=1500, d=512, L=6, H=8,
                in_dtype=cxa.CXA_F32, workspace=FAKE, workspace_bytes=BIG)

    def pop(**kw):
        a = dict(args, **kw)
        return cxa.cxa_populate(h, a["b0"], a["nb"], a["E"], a["WK"], a["WV"], a["bV"], a["T"], a["d"], a["L"],
                                a["H"], a["in_dtype"], a["workspace"], a["workspace_bytes"], 0)

    assert pop(d=500) == cxa.CXA_EINVAL                  # num_heads * head_dim != embed_dim
    assert "num_heads * head_dim" in cxa.cxa_last_error_message()
    assert pop(T=0) == cxa.CXA_EINVAL                    # positive encoder memory length
    assert pop(T=1499) == cxa.CXA_EINVAL                 # does not match the descriptor
    assert pop(b0=1, nb=2) == cxa.CXA_EINVAL             # slots out of range
    assert pop(nb=0) == cxa.CXA_EINVAL
    assert pop(E=0) == cxa.CXA_EINVAL
    assert pop(E=FAKE + 4) == cxa.CXA_EINVAL             # TMA needs 16-byte alignment
    assert pop(workspace_bytes=1024) == cxa.CXA_EINVAL
    assert pop(in_dtype=5) == cxa.CXA_EINVAL
    cxa.cxa_cache_destroy(h)


def test_invalidate_and_ready_flags(cxa_lib):
    rc, h = make(B=3)
    assert cxa.cxa_invalidate(h, -1) == cxa.CXA_OK
    assert cxa.cxa_invalidate(h, 2) == cxa.CXA_OK
    assert cxa.cxa_invalidate(h, 3) == cxa.CXA_EINVAL
    assert cxa.cxa_invalidate(h, -2) == cxa.CXA_EINVAL
    assert cxa.cxa_is_ready(h, 5) == cxa.CXA_EINVAL
    assert all(cxa.cxa_is_ready(h, b) == 0 for b in range(3))
    cxa.cxa_cache_destroy(h)


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(cxa, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        cxa.load(str(tmp_path / "missing.so"))


def test_binding_passes_explicit_streams_through():
    """An explicit stream handle (int, or an object with a cuda_stream attribute) goes to
    the C ABI unchanged; only a missing one is looked up from torch's current stream."""
    class FakeStream:
        cuda_stream = 0x1234

    assert cxa._stream(0) == 0
    assert cxa._stream(0x7f00) == 0x7f00
    assert cxa._stream(FakeStream()) == 0x1234


def test_alignment_heads_marshalled_once_per_list():
    """The (layer, head) list becomes one C int array, reused for an equal list."""
    a, n = cxa._heads_array([(3, 1), (4, 2)])
    b, m = cxa._heads_array(((3, 1), (4, 2)))
    assert n == m == 2 and a is b and list(a) == [3, 1, 4, 2]
    c, k = cxa._heads_array([])
    assert k == 0


def test_pack_weights_validates_before_any_cuda_call(cxa_lib):
    n = cxa.cxa_populate_workspace_bytes(512, 6, cxa.CXA_F32)
    assert cxa.cxa_pack_weights(FAKE, FAKE, 500, 6, cxa.CXA_F32, FAKE, n, 0) == cxa.CXA_EINVAL     # d % 64
    assert cxa.cxa_pack_weights(0, FAKE, 512, 6, cxa.CXA_F32, FAKE, n, 0) == cxa.CXA_EINVAL        # NULL WK
    assert cxa.cxa_pack_weights(FAKE, FAKE, 512, 6, 9, FAKE, n, 0) == cxa.CXA_EINVAL              # dtype
    assert cxa.cxa_pack_weights(FAKE, FAKE, 512, 6, cxa.CXA_F32, FAKE + 16, n, 0) == cxa.CXA_EINVAL  # alignment
    assert cxa.cxa_pack_weights(FAKE, FAKE, 512, 6, cxa.CXA_F32, FAKE, n - 1, 0) == cxa.CXA_EINVAL   # short
    assert "smaller" in cxa.cxa_last_error_message()


def test_populate_packed_validates_before_any_cuda_call(cxa_lib):
    rc, h = make(B=2, T=1500, L=6, H=8)
    n = cxa.cxa_populate_workspace_bytes(512, 6, cxa.CXA_F32)
    args = dict(E=FAKE, packed=FAKE, nbytes=n, bV=FAKE)

    def call(**kw):
        a = dict(args, **kw)
        return cxa.cxa_populate_packed(h, 0, 2, a["E"], a["packed"], a["nbytes"], a["bV"], 1500, 512, 6, 8,
                                       cxa.CXA_F32, 0)
    assert call(packed=0) == cxa.CXA_EINVAL
    assert call(nbytes=n - 4) == cxa.CXA_EINVAL
    assert call(E=FAKE + 4) == cxa.CXA_EINVAL
    assert cxa.cxa_populate_packed(h, 1, 2, FAKE, FAKE, n, FAKE, 1500, 512, 6, 8, cxa.CXA_F32, 0) == cxa.CXA_EINVAL
    assert cxa.cxa_populate_packed(h, 0, 2, FAKE, FAKE, n, FAKE, 1500, 512, 6, 4, cxa.CXA_F32, 0) == cxa.CXA_EINVAL
    assert cxa.cxa_is_ready(h, 0) == 0 and cxa.cxa_is_ready(h, 1) == 0
    cxa.cxa_cache_destroy(h)


def test_populate_policy_values(cxa_lib):
    for p in (cxa.CXA_POPULATE_AUTO, cxa.CXA_POPULATE_PAIR, cxa.CXA_POPULATE_SINGLE):
        assert cxa.cxa_set_populate_policy(p) == cxa.CXA_OK
    assert cxa.cxa_set_populate_policy(3) == cxa.CXA_EINVAL
    assert "unknown policy" in cxa.cxa_last_error_message()
    assert cxa.cxa_set_populate_policy(-1) == cxa.CXA_EINVAL
    assert cxa.cxa_set_populate_policy(cxa.CXA_POPULATE_AUTO) == cxa.CXA_OK


def test_decode_policy_values(cxa_lib):
    for p in (cxa.CXA_DECODE_AUTO, cxa.CXA_DECODE_STREAM, cxa.CXA_DECODE_ROWS):
        assert cxa.cxa_set_decode_policy(p) == cxa.CXA_OK
    assert cxa.cxa_set_decode_policy(3) == cxa.CXA_EINVAL
    assert cxa.cxa_set_decode_policy(-1) == cxa.CXA_EINVAL
    assert cxa.cxa_set_decode_policy(cxa.CXA_DECODE_AUTO) == cxa.CXA_OK


def test_convert_bf16_validates_before_any_cuda_call(cxa_lib):
    assert cxa.cxa_convert_bf16(0, FAKE, 8, 0) == cxa.CXA_EINVAL            # NULL source
    assert cxa.cxa_convert_bf16(FAKE, 0, 8, 0) == cxa.CXA_EINVAL            # NULL destination
    assert cxa.cxa_convert_bf16(FAKE + 4, FAKE + BIG, 8, 0) == cxa.CXA_EINVAL   # misaligned source
    assert cxa.cxa_convert_bf16(FAKE, FAKE + BIG + 2, 8, 0) == cxa.CXA_EINVAL   # misaligned destination
    assert cxa.cxa_convert_bf16(FAKE, FAKE + 16, 64, 0) == cxa.CXA_EINVAL      # overlap
    assert "overlap" in cxa.cxa_last_error_message()
    assert cxa.cxa_convert_bf16(FAKE, FAKE + BIG, 0, 0) == cxa.CXA_OK           # nothing to do, no CUDA call


def test_noalloc_rejects_unsupported_geometry_before_any_cuda_call(cxa_lib):
    # a descriptor with dh = 64 but scratch beyond the fixed maximum is refused with a
    # message naming the maximum; the check comes before any CUDA call
    rc, h = make(B=64, T=32768, L=6, H=8)
    assert rc == cxa.CXA_OK
    assert cxa.cxa_decode_noalloc(h, FAKE, FAKE, FAKE + 4096, 0.0, 0) == cxa.CXA_EINVAL
    assert "fixed maximum" in cxa.cxa_last_error_message()
    cxa.cxa_cache_destroy(h)
