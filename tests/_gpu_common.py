"""Shared helpers of the GPU parity tests (device copies of seeded inputs)."""
import json
import os

import numpy as np
import torch

from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W

# Tolerances (stated with the workloads they apply to):
POPULATE_REL_FROB = 2e-3     # populate, TF32 or bf16 tensor-core inputs, fp32 accumulate
DECODE_F32_MAX_ABS = 1e-4    # decode on an fp32 cache
DECODE_BF16_MAX_ABS = 1e-2   # decode on a bf16 cache

# Element-wise populate bound, from the arithmetic of the tensor-core GEMM:
#   |got - ref| <= c_in * A * (1 + c_store) + c_store * |ref| + 1e-6,
#   A = (|E| x |W|) (+ |bV| on V): the sum of the magnitudes of the products.
# c_in covers operand rounding and fp32 accumulation: fp32 inputs are read as TF32
# (E truncated, < 2^-10 relative; W rounded to nearest, <= 2^-11; product <= 1.47e-3)
# plus d * 2^-23 of accumulation (6e-5 at d = 512) -> 2^-9. bf16 inputs reach the
# oracle already rounded, so only the accumulation remains (d * 2^-23 = 1.5e-4 at
# d = 1280) -> 2^-11. c_store is the unit roundoff of the cache store: 2^-24 fp32,
# 2^-8 bf16 (round to nearest even, 8 significant bits).
POPULATE_C_IN = {"f32": 2.0 ** -9, "bf16": 2.0 ** -11}
POPULATE_C_STORE = {"f32": 2.0 ** -24, "bf16": 2.0 ** -8}
# Per (slot, layer, head) block: max |err| <= k * max |ref| of the block. TF32
# operands measure ~5e-4 there; a bf16 store adds up to 2^-8 of the largest value.
POPULATE_BLOCK = {"f32": 2e-3, "bf16": 5e-3}


POLICIES = {"auto": cxa.CXA_DECODE_AUTO, "stream": cxa.CXA_DECODE_STREAM, "rows": cxa.CXA_DECODE_ROWS}


POPULATE_POLICIES = {"auto": cxa.CXA_POPULATE_AUTO, "pair": cxa.CXA_POPULATE_PAIR,
                     "single": cxa.CXA_POPULATE_SINGLE}


class populate_policy:
    """Context manager: run the enclosed populates with one GEMM shape (CTA pairs
    or one CTA per tile), then go back to the automatic choice."""

    def __init__(self, name: str):
        self.code = POPULATE_POLICIES[name]

    def __enter__(self):
        assert cxa.cxa_set_populate_policy(self.code) == cxa.CXA_OK
        return self

    def __exit__(self, *exc):
        cxa.cxa_set_populate_policy(cxa.CXA_POPULATE_AUTO)
        return False


class decode_policy:
    """Context manager: run the enclosed decodes with one kernel shape (the
    persistent stream kernel or the cluster-per-row latency kernel), then go back
    to the automatic choice."""

    def __init__(self, name: str):
        self.code = POLICIES[name]

    def __enter__(self):
        assert cxa.cxa_set_decode_policy(self.code) == cxa.CXA_OK
        return self

    def __exit__(self, *exc):
        cxa.cxa_set_decode_policy(cxa.CXA_DECODE_AUTO)
        return False


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


def check_populate_block(got, ref, bound_mag, in_dtype: str, cache_dtype: str, what: str = ""):
    """Element-wise populate gate on one or more head blocks.

    got, ref, bound_mag: fp64 arrays of the same shape whose last two axes are
    (t, c) of one (slot, layer, head); bound_mag holds |E| x |W| (+ |bV|) for the
    same elements (the oracle's projection of the magnitudes). Checks every
    element against the arithmetic bound above and every block's largest error
    against POPULATE_BLOCK x its largest reference value; returns the worst
    block ratio for reporting."""
    c_in, c_st = POPULATE_C_IN[in_dtype], POPULATE_C_STORE[cache_dtype]
    err = np.abs(got - ref)
    lim = c_in * bound_mag * (1.0 + c_st) + c_st * np.abs(ref) + 1e-6
    bad = err > lim
    assert not bad.any(), (f"{what}: {int(bad.sum())} element(s) beyond the arithmetic bound, first at "
                           f"{tuple(int(i) for i in np.argwhere(bad)[0])}: err {err[bad][0]:.3e} > {lim[bad][0]:.3e}")
    blk_err = err.max(axis=(-2, -1))
    blk_ref = np.abs(ref).max(axis=(-2, -1))
    ratio = blk_err / np.maximum(blk_ref, 1e-30)
    worst = float(ratio.max())
    assert worst <= POPULATE_BLOCK[cache_dtype], f"{what}: a head block's max error is {worst:.3e} of its max value"
    return worst


def check_populate(Kg, Vg, E, WK, WV, bV, H, in_dtype: str, cache_dtype: str, what: str = ""):
    """The populate gates on whole slots: relative Frobenius <= POPULATE_REL_FROB
    over the slots given, and the element-wise / per-block gates of
    check_populate_block on every (slot, layer, head) block. Kg, Vg: the GPU
    cache of those slots as fp64 [nb, L, H, T, dh]; E [nb, T, d] and the weights
    as the oracle takes them. One slot at a time keeps host memory small.
    Returns (rel-Frobenius K, rel-Frobenius V, worst block ratio)."""
    from oracle import cross_attention as O
    nb = E.shape[0]
    num = {"K": 0.0, "V": 0.0}
    den = {"K": 0.0, "V": 0.0}
    aWK, aWV, abV = np.abs(np.asarray(WK, np.float64)), np.abs(np.asarray(WV, np.float64)), np.abs(np.asarray(bV, np.float64))
    worst = 0.0
    for b in range(nb):
        Kr, Vr = O.populate(E[b:b + 1], WK, WV, bV, H)
        Ka, Va = O.populate(np.abs(np.asarray(E[b:b + 1], np.float64)), aWK, aWV, abV, H)
        for name, got, ref, mag in (("K", Kg[b:b + 1], Kr, Ka), ("V", Vg[b:b + 1], Vr, Va)):
            num[name] += float(((got - ref) ** 2).sum())
            den[name] += float((ref ** 2).sum())
            worst = max(worst, check_populate_block(got, ref, mag, in_dtype, cache_dtype, f"{what} slot {b} {name}"))
    fk, fv = (num["K"] / den["K"]) ** 0.5, (num["V"] / den["V"]) ** 0.5
    assert fk <= POPULATE_REL_FROB and fv <= POPULATE_REL_FROB, (what, fk, fv)
    return fk, fv, worst


def check_populate_head(Kg, Vg, E_b, WK_l, WV_l, bV_l, h: int, in_dtype: str, cache_dtype: str, what: str = ""):
    """The populate gates on one sampled (slot, layer, head) block, for workloads
    too large to project whole in fp64: relative Frobenius, element-wise bound and
    block bound against the oracle's projection of that head's columns."""
    from oracle import cross_attention as O
    Kr, Vr = O.populate_head(E_b, WK_l, WV_l, bV_l, h)
    Ka, Va = O.populate_head(np.abs(np.asarray(E_b, np.float64)), np.abs(np.asarray(WK_l, np.float64)),
                             np.abs(np.asarray(WV_l, np.float64)), np.abs(np.asarray(bV_l, np.float64)), h)
    fk, fv = O.rel_frobenius(Kg, Kr), O.rel_frobenius(Vg, Vr)
    assert fk <= POPULATE_REL_FROB and fv <= POPULATE_REL_FROB, (what, fk, fv)
    worst = max(check_populate_block(Kg, Kr, Ka, in_dtype, cache_dtype, what + " K"),
                check_populate_block(Vg, Vr, Va, in_dtype, cache_dtype, what + " V"))
    return fk, fv, worst, Kr, Vr


def record_parity(config: str, variant: str, **metrics):
    """Append one JSON line of measured errors for a (config, variant) to the file
    named by CXA_PARITY_RECORD, when it is set (a record of the parity run)."""
    path = os.environ.get("CXA_PARITY_RECORD")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"config": config, "variant": variant,
                            **{k: (float(v) if isinstance(v, (int, float, np.floating)) else v)
                               for k, v in metrics.items()}}) + "\n")
