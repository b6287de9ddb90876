"""Python binding of libcxa (include/cxa.h): argument marshalling only.

The C-named functions (``cxa_populate``, ``cxa_decode``, ``cxa_invalidate``, ...)
take raw device pointers or torch tensors (their ``data_ptr()`` is passed) and
return the C status code. ``CrossAttentionCache`` is a convenience owner of the
cache, workspaces and descriptor that raises ``CxaError`` on a non-zero status.
PyTorch is used for device memory and streams only; every step of populate and
decode runs in libcxa's CUDA kernels. There is no fallback: if the library is
not built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

CXA_OK, CXA_EINVAL, CXA_ENOTREADY, CXA_ECUDA, CXA_ETIMEOUT = 0, -1, -2, -3, -4
CXA_F32, CXA_BF16 = 0, 1
CXA_DECODE_AUTO, CXA_DECODE_STREAM, CXA_DECODE_ROWS = 0, 1, 2
CXA_POPULATE_AUTO, CXA_POPULATE_PAIR, CXA_POPULATE_SINGLE = 0, 1, 2

# every symbol include/cxa.h declares: name -> (restype, argtypes)
_c_void_pp = ctypes.POINTER(ctypes.c_void_p)
SIGNATURES = {
    "cxa_cache_create": (ctypes.c_int, [_c_void_pp, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "cxa_cache_destroy": (None, [ctypes.c_void_p]),
    "cxa_populate_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "cxa_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 5),
    "cxa_populate": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "cxa_pack_weights": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "cxa_populate_packed": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "cxa_convert_bf16": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "cxa_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "cxa_invalidate": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "cxa_is_ready": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "cxa_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "cxa_last_error_message": (ctypes.c_char_p, []),
    "cxa_launch_count": (ctypes.c_ulonglong, []),
    "cxa_device_status": (ctypes.c_int, [ctypes.c_int]),
    "cxa_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint, ctypes.c_void_p]),
    "cxa_set_decode_policy": (ctypes.c_int, [ctypes.c_int]),
    "cxa_set_populate_policy": (ctypes.c_int, [ctypes.c_int]),
    "cxa_decode_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_float, ctypes.c_void_p]),
    "cxa_decode_shared_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 6),
    "cxa_decode_shared": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_void_p]),
    "cxa_decode_layers": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p]),
    "cxa_cross_block_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 5),
    "cxa_cross_block": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                       ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "cxa_cache_append": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p]),
    "cxa_self_attention_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                               ctypes.c_size_t, ctypes.c_void_p]),
    "cxa_alignment_weights": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                             ctypes.c_void_p]),
}

# most query rows cxa_decode_shared takes per cache row (CXA_MAX_SHARED_QUERIES)
CXA_MAX_SHARED_QUERIES = 16

# bytes of the fixed device scratch behind cxa_decode_noalloc (CXA_NOALLOC_SCRATCH_BYTES)
CXA_NOALLOC_SCRATCH_BYTES = 8 << 20

_lib = None


def load(path: str | None = None):
    """Load libcxa.so (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libcxa is not built ({path} is missing); build it with "
                           "encoder_decoder_speech_gb300._build.build_library()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class CxaError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = load()
        self.code = code
        super().__init__(f"{where}: {lib.cxa_strerror(code).decode()}: {lib.cxa_last_error_message().decode()}")


def check(code: int, where: str = "cxa") -> None:
    if code != CXA_OK:
        raise CxaError(code, where)


def _ptr(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s) -> int | None:
    if s is None:
        import torch
        # the current stream's handle without building a Stream object (a few
        # microseconds per call on the host otherwise)
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


# ---------------------------------------------------------------- C-named calls
def cxa_cache_create(Kc, Vc, B, T, L, H, dh, cache_dtype):
    """Returns (status, handle); handle is None unless status == CXA_OK."""
    h = ctypes.c_void_p()
    rc = load().cxa_cache_create(ctypes.byref(h), _ptr(Kc), _ptr(Vc), B, T, L, H, dh, cache_dtype)
    return rc, (h.value if rc == CXA_OK else None)


def cxa_cache_destroy(handle) -> None:
    load().cxa_cache_destroy(handle)


def cxa_populate_workspace_bytes(d, L, in_dtype) -> int:
    return load().cxa_populate_workspace_bytes(d, L, in_dtype)


def cxa_decode_workspace_bytes(B, T, L, H, dh=64) -> int:
    return load().cxa_decode_workspace_bytes(B, T, L, H, dh)


def cxa_populate(handle, b0, nb, E, WK, WV, bV, T, d, L, H, in_dtype, workspace, workspace_bytes, stream=None) -> int:
    return load().cxa_populate(handle, b0, nb, _ptr(E), _ptr(WK), _ptr(WV), _ptr(bV), T, d, L, H, in_dtype,
                               _ptr(workspace), workspace_bytes, _stream(stream))


def cxa_pack_weights(WK, WV, d, L, in_dtype, packed, packed_bytes, stream=None) -> int:
    return load().cxa_pack_weights(_ptr(WK), _ptr(WV), d, L, in_dtype, _ptr(packed), packed_bytes, _stream(stream))


def cxa_populate_packed(handle, b0, nb, E, packed, packed_bytes, bV, T, d, L, H, in_dtype, stream=None) -> int:
    return load().cxa_populate_packed(handle, b0, nb, _ptr(E), _ptr(packed), packed_bytes, _ptr(bV), T, d, L, H,
                                      in_dtype, _stream(stream))


def cxa_convert_bf16(src, dst, n, stream=None) -> int:
    return load().cxa_convert_bf16(_ptr(src), _ptr(dst), n, _stream(stream))


def to_bf16(x, out=None, stream=None):
    """fp32 device tensor -> bf16 device tensor of the same shape (cxa_convert_bf16)."""
    import torch
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("to_bf16 takes a contiguous float32 tensor")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    check(cxa_convert_bf16(x, out, x.numel(), stream), "cxa_convert_bf16")
    return out


def cxa_decode(handle, Q, key_len, out, scale, workspace, workspace_bytes, stream=None) -> int:
    return load().cxa_decode(handle, _ptr(Q), _ptr(key_len), _ptr(out), float(scale), _ptr(workspace),
                             workspace_bytes, _stream(stream))


def cxa_decode_shared_workspace_bytes(B, T, L, H, dh=64, nq=1) -> int:
    return load().cxa_decode_shared_workspace_bytes(B, T, L, H, dh, nq)


def cxa_decode_shared(handle, nq, Q, key_len, out, scale, workspace, workspace_bytes, stream=None) -> int:
    return load().cxa_decode_shared(handle, nq, _ptr(Q), _ptr(key_len), _ptr(out), float(scale), _ptr(workspace),
                                    workspace_bytes, _stream(stream))


def cxa_decode_layers(handle, l0, nl, Q, key_len, out, scale, workspace, workspace_bytes, stream=None) -> int:
    return load().cxa_decode_layers(handle, l0, nl, _ptr(Q), _ptr(key_len), _ptr(out), float(scale),
                                    _ptr(workspace), workspace_bytes, _stream(stream))


def cxa_cross_block_workspace_bytes(B, T, L, H, dh=64) -> int:
    return load().cxa_cross_block_workspace_bytes(B, T, L, H, dh)


def cxa_cross_block(handle, layer, x, ln_gamma, ln_beta, ln_eps, WQ, bQ, WO, bO, key_len, scale, workspace,
                    workspace_bytes, stream=None) -> int:
    return load().cxa_cross_block(handle, layer, _ptr(x), _ptr(ln_gamma), _ptr(ln_beta), float(ln_eps), _ptr(WQ),
                                  _ptr(bQ), _ptr(WO), _ptr(bO), _ptr(key_len), float(scale), _ptr(workspace),
                                  workspace_bytes, _stream(stream))


def cxa_cache_append(handle, pos, K_new, V_new, stream=None) -> int:
    return load().cxa_cache_append(handle, _ptr(pos), _ptr(K_new), _ptr(V_new), _stream(stream))


def cxa_self_attention_step(handle, pos, Q, K_new, V_new, out, scale, workspace, workspace_bytes, stream=None) -> int:
    return load().cxa_self_attention_step(handle, _ptr(pos), _ptr(Q), _ptr(K_new), _ptr(V_new), _ptr(out), float(scale),
                                          _ptr(workspace), workspace_bytes, _stream(stream))


_HEADS_ARRAYS: dict = {}


def _heads_array(heads):
    """The (layer, head) pairs as a C int array, kept per distinct head list (a call
    site passes the same list every step)."""
    key = tuple((int(l), int(h)) for l, h in heads)
    arr = _HEADS_ARRAYS.get(key)
    if arr is None:
        flat = [v for pair in key for v in pair]
        arr = (ctypes.c_int * max(len(flat), 1))(*flat)
        if len(_HEADS_ARRAYS) < 256:
            _HEADS_ARRAYS[key] = arr
    return arr, len(key)


def cxa_alignment_weights(handle, Q, key_len, heads, weights, mean, scale, stream=None) -> int:
    """heads: host sequence of (layer, head) pairs."""
    arr, n = _heads_array(heads)
    return load().cxa_alignment_weights(handle, _ptr(Q), _ptr(key_len), ctypes.cast(arr, ctypes.c_void_p), n,
                                        _ptr(weights), _ptr(mean), float(scale), _stream(stream))


def cxa_decode_noalloc(handle, Q, key_len, out, scale, stream=None) -> int:
    """cxa_decode with its scratch in libcxa's fixed device array: for callers
    that cannot allocate device memory. Calls must be ordered on one stream."""
    return load().cxa_decode_noalloc(handle, _ptr(Q), _ptr(key_len), _ptr(out), float(scale), _stream(stream))


def cxa_invalidate(handle, b=-1) -> int:
    return load().cxa_invalidate(handle, b)


def cxa_is_ready(handle, b) -> int:
    return load().cxa_is_ready(handle, b)


def cxa_strerror(code) -> str:
    return load().cxa_strerror(code).decode()


def cxa_last_error_message() -> str:
    return load().cxa_last_error_message().decode()


def cxa_launch_count() -> int:
    return load().cxa_launch_count()


def cxa_device_status(clear=0) -> int:
    return load().cxa_device_status(clear)


def cxa_set_decode_policy(policy: int) -> int:
    """Process-wide choice of the one-query decode kernel shape (CXA_DECODE_*)."""
    return load().cxa_set_decode_policy(policy)


def cxa_set_populate_policy(policy: int) -> int:
    """Process-wide choice of the populate GEMM shape (CXA_POPULATE_*)."""
    return load().cxa_set_populate_policy(policy)


def cxa_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    """Enqueue the bounded-wait self-test kernel (its wait expires after limit_us)."""
    return load().cxa_selftest_wait_timeout(limit_us, _stream(stream))


# ---------------------------------------------------------------- owner object
_DTYPES = {"f32": CXA_F32, "bf16": CXA_BF16}


def _dtype_code(t) -> int:
    import torch
    if t == torch.float32:
        return CXA_F32
    if t == torch.bfloat16:
        return CXA_BF16
    raise TypeError(f"unsupported dtype {t}; expected float32 or bfloat16")


class CrossAttentionCache:
    """Owns a [B][L][H][T][64] K/V projection cache, its decode workspace and
    the libcxa descriptor; allocation goes through torch on ``device``."""

    def __init__(self, B: int, T: int, L: int, H: int, dh: int = 64, cache_dtype: str = "f32", device="cuda"):
        import torch
        self.B, self.T, self.L, self.H, self.dh = B, T, L, H, dh
        self.d = H * dh
        self.cache_dtype = cache_dtype
        tdt = torch.float32 if cache_dtype == "f32" else torch.bfloat16
        self.Kc = torch.empty((B, L, H, T, dh), dtype=tdt, device=device)
        self.Vc = torch.empty((B, L, H, T, dh), dtype=tdt, device=device)
        self.decode_ws_bytes = cxa_decode_workspace_bytes(B, T, L, H, dh)
        self.decode_ws = torch.zeros(max(self.decode_ws_bytes, 256), dtype=torch.uint8, device=device)
        self._pop_ws = {}
        self._shared_ws = None
        self._block_ws = None
        rc, h = cxa_cache_create(self.Kc, self.Vc, B, T, L, H, dh, _DTYPES[cache_dtype])
        check(rc, "cxa_cache_create")
        self.handle = h

    def populate_workspace(self, in_dtype: int):
        import torch
        if in_dtype not in self._pop_ws:
            n = cxa_populate_workspace_bytes(self.d, self.L, in_dtype)
            self._pop_ws[in_dtype] = torch.empty(n, dtype=torch.uint8, device=self.Kc.device)
        return self._pop_ws[in_dtype]

    def populate(self, E, WK, WV, bV, b0: int = 0, stream=None) -> None:
        """E [nb, T, d]; WK, WV [L, d, d] (d_in, d_out), same dtype as E; bV [L, d] fp32."""
        in_dtype = _dtype_code(E.dtype)
        for name, t in (("E", E), ("WK", WK), ("WV", WV), ("bV", bV)):
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if WK.dtype != E.dtype or WV.dtype != E.dtype:
            raise TypeError("WK and WV must have E's dtype")
        nb = E.shape[0] if E.dim() == 3 else 1
        ws = self.populate_workspace(in_dtype)
        check(cxa_populate(self.handle, b0, nb, E, WK, WV, bV, E.shape[-2], E.shape[-1], WK.shape[0],
                           self.H, in_dtype, ws, ws.numel(), stream), "cxa_populate")

    def pack_weights(self, WK, WV, stream=None):
        """Pack WK, WV [L, d, d] (d_in, d_out) once for populate_packed; returns the
        packed buffer (a uint8 device tensor owned by the caller)."""
        import torch
        in_dtype = _dtype_code(WK.dtype)
        if WV.dtype != WK.dtype or not WK.is_contiguous() or not WV.is_contiguous():
            raise ValueError("WK and WV must be contiguous and of one dtype")
        n = cxa_populate_workspace_bytes(self.d, self.L, in_dtype)
        packed = torch.empty(n, dtype=torch.uint8, device=self.Kc.device)
        check(cxa_pack_weights(WK, WV, self.d, self.L, in_dtype, packed, n, stream), "cxa_pack_weights")
        return packed

    def populate_packed(self, E, packed, bV, b0: int = 0, stream=None) -> None:
        """E [nb, T, d] (fp32 or bf16, the dtype the weights were packed in); bV [L, d] fp32."""
        in_dtype = _dtype_code(E.dtype)
        if not E.is_contiguous() or not bV.is_contiguous():
            raise ValueError("E and bV must be contiguous")
        nb = E.shape[0] if E.dim() == 3 else 1
        check(cxa_populate_packed(self.handle, b0, nb, E, packed, packed.numel(), bV, E.shape[-2], E.shape[-1],
                                  self.L, self.H, in_dtype, stream), "cxa_populate_packed")

    def decode(self, Q, key_len, out=None, scale: float = 0.0, stream=None):
        """Q [B, L, H, 64] fp32, key_len [B] int32 (device). Returns out [B, L, H, 64] fp32."""
        import torch
        if out is None:
            out = torch.empty_like(Q)
        check(cxa_decode(self.handle, Q, key_len, out, scale, self.decode_ws, self.decode_ws_bytes, stream),
              "cxa_decode")
        return out

    def decode_shared(self, Q, key_len, out=None, scale: float = 0.0, stream=None):
        """Q [B, nq, L, H, 64] fp32: nq hypotheses per slot sharing the slot's cache.
        Returns out [B, nq, L, H, 64] fp32."""
        import torch
        nq = Q.shape[1]
        need = cxa_decode_shared_workspace_bytes(self.B, self.T, self.L, self.H, self.dh, nq)
        if self._shared_ws is None or self._shared_ws.numel() < need:
            self._shared_ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.Kc.device)
        if out is None:
            out = torch.empty_like(Q)
        check(cxa_decode_shared(self.handle, nq, Q, key_len, out, scale, self._shared_ws, self._shared_ws.numel(),
                                stream), "cxa_decode_shared")
        return out

    def decode_layers(self, l0: int, Q, key_len, out=None, scale: float = 0.0, stream=None):
        """Q [B, nl, H, 64] fp32 for layers [l0, l0+nl). Returns out of the same shape."""
        import torch
        if out is None:
            out = torch.empty_like(Q)
        check(cxa_decode_layers(self.handle, l0, Q.shape[1], Q, key_len, out, scale, self.decode_ws,
                                self.decode_ws_bytes, stream), "cxa_decode_layers")
        return out

    def cross_block(self, layer: int, x, WQ, WO, key_len, ln_gamma=None, ln_beta=None, ln_eps: float = 1e-5,
                    bQ=None, bO=None, scale: float = 0.0, stream=None):
        """One decoder layer's cross-attention block, in place on x [B, d] fp32."""
        import torch
        need = cxa_cross_block_workspace_bytes(self.B, self.T, self.L, self.H, self.dh)
        if self._block_ws is None or self._block_ws.numel() < need:
            self._block_ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.Kc.device)
        check(cxa_cross_block(self.handle, layer, x, ln_gamma, ln_beta, ln_eps, WQ, bQ, WO, bO, key_len, scale,
                              self._block_ws, self._block_ws.numel(), stream), "cxa_cross_block")
        return x

    def append(self, pos, K_new, V_new, stream=None) -> None:
        """Write K_new/V_new [B, L, H, 64] fp32 at position pos[b] (device int32 [B])."""
        check(cxa_cache_append(self.handle, pos, K_new, V_new, stream), "cxa_cache_append")

    def self_attention_step(self, pos, Q, K_new, V_new, out=None, scale: float = 0.0, stream=None):
        """Append the new rows at pos, then decode Q over positions 0 .. pos[b]."""
        import torch
        if out is None:
            out = torch.empty_like(Q)
        check(cxa_self_attention_step(self.handle, pos, Q, K_new, V_new, out, scale, self.decode_ws,
                                      self.decode_ws_bytes, stream), "cxa_self_attention_step")
        return out

    def alignment_weights(self, Q, key_len, heads, scale: float = 0.0, with_mean: bool = True, stream=None):
        """Softmax rows [B, nsel, T] of the (layer, head) pairs in `heads` for queries
        Q [B, L, H, 64], and their mean over heads [B, T] (or None)."""
        import torch
        w = torch.empty((self.B, len(heads), self.T), dtype=torch.float32, device=self.Kc.device)
        m = torch.empty((self.B, self.T), dtype=torch.float32, device=self.Kc.device) if with_mean else None
        check(cxa_alignment_weights(self.handle, Q, key_len, heads, w, m, scale, stream), "cxa_alignment_weights")
        return w, m

    def invalidate(self, b: int = -1) -> None:
        check(cxa_invalidate(self.handle, b), "cxa_invalidate")

    def is_ready(self, b: int) -> bool:
        return cxa_is_ready(self.handle, b) == 1

    def close(self) -> None:
        if getattr(self, "handle", None):
            cxa_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
