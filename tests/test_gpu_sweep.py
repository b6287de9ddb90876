"""Parity on the decode bandwidth sweep workload (d = 512, 8 heads x 64, 6
layers; E and W ~ N(0, 1/d); key_len = T) at its corners, up to the largest
point T = 32768, B = 64 (a 51.5 GB fp32 cache). Sampled (slot, layer, head)
K/V blocks are compared with the oracle's projection and sampled decode rows
with the oracle on the GPU's own cache, in the launch configuration the
benchmark uses."""
import numpy as np
import pytest
import torch

from _gpu_common import DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, check_populate_head, dev, host, record_parity
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


@pytest.mark.parametrize("T,B", [(256, 64), (1500, 4), (4096, 16), (16384, 1), (32768, 64)])
def test_sweep_point(T, B):
    w = W.sweep_workload(T, B)
    WK, WV, bV = W.make_weights(w)
    kl = W.make_key_len(w)
    E = torch.empty((B, T, w.d), dtype=torch.float32, device="cuda")
    for b in range(B):                     # one memory at a time keeps host memory small
        E[b].copy_(torch.from_numpy(W.make_E(w, b, kl)))
    rng = np.random.default_rng(T + B)
    picks = sorted({(int(rng.integers(B)), int(rng.integers(w.L)), int(rng.integers(w.H))) for _ in range(6)}
                   | {(0, 0, 0), (B - 1, w.L - 1, w.H - 1)})
    Q = W.make_Q(w, 0)
    for cache_dtype in ("f32", "bf16"):
        c = cxa.CrossAttentionCache(B, T, w.L, w.H, 64, cache_dtype)
        c.populate(E, dev(WK), dev(WV), dev(bV))
        out = host(c.decode(dev(Q), dev(kl, torch.int32)))
        wf = wb = wi = 0.0
        for (b, l, h) in picks:
            Kg, Vg = host(c.Kc[b, l, h]), host(c.Vc[b, l, h])
            fk, fv, blk, _, _ = check_populate_head(Kg, Vg, W.make_E(w, b, kl), WK[l], WV[l], bV[l], h, "f32",
                                                    cache_dtype, f"sweep T{T} B{B} ({b}, {l}, {h})")
            iso = O.attend_row(Q[b, l, h], Kg, Vg, int(kl[b]), w.scale)
            wf, wb, wi = max(wf, fk, fv), max(wb, blk), max(wi, np.abs(out[b, l, h] - iso).max())
            assert np.abs(out[b, l, h] - iso).max() <= TOL[cache_dtype]
        record_parity(f"sweep T{T} B{B}", f"{cache_dtype} cache", sampled_heads=len(picks),
                      populate_worst_rel_frob=wf, populate_worst_block_ratio=wb, decode_max_abs_kernel_isolated=wi)
        c.close()
        del c
        torch.cuda.empty_cache()
