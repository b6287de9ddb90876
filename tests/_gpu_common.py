"""Shared helpers of the GPU parity tests (device copies of seeded inputs)."""
import numpy as np
import torch

from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W

# Tolerances (stated with the workloads they apply to):
POPULATE_REL_FROB = 2e-3     # populate, TF32 or bf16 tensor-core inputs, fp32 accumulate
DECODE_F32_MAX_ABS = 1e-4    # decode on an fp32 cache
DECODE_BF16_MAX_ABS = 1e-2   # decode on a bf16 cache


def dev(x, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=dtype)


def inputs_on_device(w: W.Workload):
    """Seeded E, WK, WV, bV, key_len for workload w, on the GPU in w's input dtype,
    plus the same values on the host (float32 arrays, bf16-exact for bf16 inputs)."""
    E = W.make_E_all(w)
    WK, WV, bV = W.make_weights(w)
    kl = W.make_key_len(w)
    tdt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    d = dict(E=dev(E, tdt), WK=dev(WK, tdt), WV=dev(WV, tdt), bV=dev(bV), key_len=dev(kl, torch.int32))
    h = dict(E=E, WK=WK, WV=WV, bV=bV, key_len=kl)
    return d, h


def cache_for(w: W.Workload, cache_dtype: str):
    return cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, cache_dtype)


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
