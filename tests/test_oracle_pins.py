"""Pins for the fp64 oracle: brute force, closed forms, the invariants the pages
fix, and the printed Whisper-Base layout facts. Each pin is also run against
deliberately broken copies of the oracle (planted on the CPU) to show that a
plausible mistake -- a transposed operand, a wrong sign, a dropped term, an
off-by-one mask, a wrong layout -- makes at least one pin fail.
"""
import json
import math
import os

import numpy as np
import pytest

from encoder_decoder_speech_gb300 import workloads as W
from oracle import cross_attention as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "whisper_base_decode_call.json")


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


# ---------------------------------------------------------------------------
# independent pure-Python restatements (no numpy arithmetic, fsum sums)
# ---------------------------------------------------------------------------
def bf_populate(E, WK, WV, bV, H):
    """K[b][l][h][t][c] = sum_i E[b][t][i] * WK[l][i][h*dh+c]; V adds bV[l][h*dh+c]."""
    E, WK, WV, bV = E.tolist(), WK.tolist(), WV.tolist(), bV.tolist()
    B, T, d, L = len(E), len(E[0]), len(E[0][0]), len(WK)
    dh = d // H
    K = [[[[[0.0] * dh for _ in range(T)] for _ in range(H)] for _ in range(L)] for _ in range(B)]
    V = [[[[[0.0] * dh for _ in range(T)] for _ in range(H)] for _ in range(L)] for _ in range(B)]
    for b in range(B):
        for l in range(L):
            for h in range(H):
                for t in range(T):
                    for c in range(dh):
                        j = h * dh + c
                        K[b][l][h][t][c] = math.fsum(E[b][t][i] * WK[l][i][j] for i in range(d))
                        V[b][l][h][t][c] = math.fsum([E[b][t][i] * WV[l][i][j] for i in range(d)]
                                                     + [bV[l][j]])
    return np.array(K), np.array(V)


def bf_attend(q, K, V, n, scale):
    """softmax without the max shift: w_t = exp(s_t) / sum_u exp(s_u)."""
    q, K, V = list(q), [list(r) for r in K], [list(r) for r in V]
    dh = len(q)
    if n <= 0:
        return [0.0] * dh
    e = [math.exp(scale * math.fsum(q[c] * K[t][c] for c in range(dh))) for t in range(n)]
    z = math.fsum(e)
    return [math.fsum(e[t] * V[t][c] for t in range(n)) / z for c in range(dh)]


# ---------------------------------------------------------------------------
# pin checks, each returning an error measure (0 == exact agreement)
# ---------------------------------------------------------------------------
def pin_populate_bruteforce():
    err = 0.0
    for (B, T, d, L, H) in [(2, 1, 4, 2, 2), (1, 2, 4, 2, 2), (2, 3, 4, 1, 2), (1, 3, 6, 2, 3)]:
        E, WK, WV = _rand((B, T, d), 1), _rand((L, d, d), 2), _rand((L, d, d), 3)
        bV = _rand((L, d), 4)
        Kc, Vc = O.populate(E, WK, WV, bV, H)
        Kb, Vb = bf_populate(E, WK, WV, bV, H)
        err = max(err, np.abs(Kc - Kb).max(), np.abs(Vc - Vb).max())
    return err


def pin_decode_bruteforce():
    err = 0.0
    cases = [(1, 2, 2, 1), (2, 2, 2, 2), (3, 2, 2, 3), (3, 2, 2, 2), (5, 64, 1, 5), (5, 64, 1, 3), (4, 2, 2, 0)]
    for i, (T, dh, H, n) in enumerate(cases):
        B, L = 2, 2
        Q = _rand((B, L, H, dh), 10 + i)
        Kc = _rand((B, L, H, T, dh), 20 + i)
        Vc = _rand((B, L, H, T, dh), 30 + i)
        kl = np.array([n, T])
        scale = 1.0 / math.sqrt(dh)
        out = O.decode(Q, Kc, Vc, kl, scale)
        for b in range(B):
            for l in range(L):
                for h in range(H):
                    ref = bf_attend(Q[b, l, h], Kc[b, l, h], Vc[b, l, h], int(kl[b]), scale)
                    err = max(err, float(np.abs(out[b, l, h] - np.array(ref)).max()))
    return err


def pin_closed_forms():
    """Returns the largest deviation from the closed forms."""
    errs = []
    B, L, H, T, dh = 2, 2, 2, 9, 64
    Q = _rand((B, L, H, dh), 40)
    Kc, Vc = _rand((B, L, H, T, dh), 41), _rand((B, L, H, T, dh), 42)
    # key_len = 1 (or T = 1): the output is V row 0
    out = O.decode(Q, Kc, Vc, [1, 1])
    errs.append(np.abs(out - Vc[:, :, :, 0]).max())
    out = O.decode(Q, Kc[:, :, :, :1], Vc[:, :, :, :1], [1, 1])
    errs.append(np.abs(out - Vc[:, :, :, 0]).max())
    # q = 0: uniform weights -> mean of the first n V rows
    out = O.decode(np.zeros_like(Q), Kc, Vc, [5, 9])
    errs.append(np.abs(out[0] - Vc[0, :, :, :5].mean(axis=2)).max())
    errs.append(np.abs(out[1] - Vc[1].mean(axis=2)).max())
    # V rows all equal to one vector -> that vector
    vconst = _rand((dh,), 43)
    out = O.decode(Q, Kc, np.broadcast_to(vconst, Vc.shape), [9, 4])
    errs.append(np.abs(out - vconst).max())
    # one key aligned with q by a huge margin, another anti-aligned: the output is
    # the aligned key's V row (a flipped softmax sign would pick the other one)
    K2 = Kc * 1e-3
    for b in range(B):
        for l in range(L):
            for h in range(H):
                qn = Q[b, l, h] / np.linalg.norm(Q[b, l, h])
                K2[b, l, h, 3] = 60.0 * qn
                K2[b, l, h, 6] = -60.0 * qn
    out = O.decode(Q, K2, Vc, [9, 9], scale=1.0)
    errs.append(np.abs(out - Vc[:, :, :, 3]).max())
    # key_len = 0 -> zeros; key_len beyond T clamps to T; negative clamps to 0
    out = O.decode(Q, Kc, Vc, [0, 100])
    errs.append(np.abs(out[0]).max())
    errs.append(np.abs(out[1] - O.decode(Q, Kc, Vc, [T, T])[1]).max())
    errs.append(np.abs(O.decode(Q, Kc, Vc, [-3, 0])).max())
    return float(max(errs))


def pin_key_bias_invariance():
    """Adding a key bias bK leaves decode unchanged (WhisperKit case study §2)."""
    B, T, d, L, H = 2, 11, 128, 2, 2
    E, WK, WV, bV = _rand((B, T, d), 50), _rand((L, d, d), 51, d ** -0.5), _rand((L, d, d), 52, d ** -0.5), _rand((L, d), 53, 0.02)
    bK = _rand((L, d), 54)
    Q = _rand((B, L, H, 64), 55)
    Kc, Vc = O.populate(E, WK, WV, bV, H)
    Kb, Vb = O.populate(E, WK, WV, bV, H, bK=bK)
    assert np.abs(Kb - Kc).max() > 0.1            # the bias really changed the keys
    a = O.decode(Q, Kc, Vc, [11, 7])
    c = O.decode(Q, Kb, Vb, [11, 7])
    return float(np.abs(a - c).max() / np.abs(a).max())


def pin_full_window():
    """One-query decode == the matching row of the full-window formula
    ("Recurrence as feeds": the whole-window formula kept as a check)."""
    B, T, L, H, dh = 1, 13, 1, 1, 64
    Kc, Vc = _rand((B, L, H, T, dh), 60), _rand((B, L, H, T, dh), 61)
    Qblock = _rand((7, dh), 62)
    err = 0.0
    for n in (13, 8):
        full = O.full_window(Qblock, Kc[0, 0, 0], Vc[0, 0, 0], n, 0.125)
        for r in range(7):
            one = O.decode(Qblock[r].reshape(1, 1, 1, dh), Kc, Vc, [n])[0, 0, 0]
            err = max(err, float(np.abs(one - full[r]).max() / np.abs(full[r]).max()))
    return err


def pin_cache_reuse():
    """4 decode steps on one populated cache == re-projecting E every step
    ("View 3 -- prefill vs decode": projected once, reused per step)."""
    w = W.custom("reuse", B=2, T=17, d=128, L=2, H=2, ragged=True, steps=4)
    E, (WK, WV, bV), kl = W.make_E_all(w), W.make_weights(w), W.make_key_len(w)
    Kc, Vc = O.populate(E, WK, WV, bV, w.H)
    err = 0.0
    for s in range(4):
        Q = W.make_Q(w, s)
        err = max(err, float(np.abs(O.decode(Q, Kc, Vc, kl)
                                    - O.cross_attention_from_memory(Q, E, WK, WV, bV, kl, w.H)).max()))
    return err


def pin_layout_offset():
    """Whisper-Base dims: the layer-5 K slab starts 15,360,000 bytes into an fp32
    cache, and element (l, h, t, c) sits at ((l*H + h)*T + t)*dh + c."""
    g = json.load(open(GOLDEN))
    T, d = g["encoder_memory_shape"]
    L, H, dh = g["decoder_layers"], g["num_heads"], g["head_dim"]
    E = _rand((1, T, d), 70)
    WK, WV = _rand((L, d, d), 71, d ** -0.5), _rand((L, d, d), 72, d ** -0.5)
    Kc, _ = O.populate(E, WK, WV, np.zeros((L, d)), H)
    flat = Kc.reshape(-1)
    bad = 0
    idx = g["layer5_k_cache_offset_bytes"] // 4
    if not np.isclose(flat[idx], E[0, 0] @ WK[5][:, 0], rtol=1e-12, atol=1e-12):
        bad += 1
    for (l, h, t, c) in [(5, 0, 0, 0), (5, 3, 7, 11), (2, 7, 1499, 63), (0, 1, 1, 0)]:
        if not np.isclose(flat[((l * H + h) * T + t) * dh + c], E[0, t] @ WK[l][:, h * dh + c],
                          rtol=1e-12, atol=1e-12):
            bad += 1
    return bad


def pin_token_major_rejected():
    """A token-major cache has the same element count but must not decode to the
    same result ("Deliberate failure": shape equality is not compatibility)."""
    w = W.custom("tm", B=1, T=12, d=128, L=2, H=2)
    E, (WK, WV, bV) = W.make_E_all(w), W.make_weights(w)
    Kc, Vc = O.populate(E, WK, WV, bV, w.H)
    tok_K = np.stack([E[0] @ WK[l] for l in range(w.L)]).reshape(Kc.shape)
    tok_V = np.stack([E[0] @ WV[l] + bV[l] for l in range(w.L)]).reshape(Vc.shape)
    Q = W.make_Q(w, 0)
    good = O.decode(Q, Kc, Vc, [12])
    wrong = O.decode(Q, tok_K, tok_V, [12])
    return float(np.abs(good - wrong).max())


def pin_scale_on_scores():
    """scale multiplies q.k: decode(Q, scale=s) == decode(s*Q, scale=1); default 1/sqrt(dh)."""
    B, L, H, T, dh = 1, 2, 2, 10, 64
    Q, Kc, Vc = _rand((B, L, H, dh), 80), _rand((B, L, H, T, dh), 81), _rand((B, L, H, T, dh), 82)
    a = O.decode(Q, Kc, Vc, [10], scale=0.37)
    b = O.decode(0.37 * Q, Kc, Vc, [10], scale=1.0)
    c = O.decode(Q, Kc, Vc, [10])
    d = O.decode(Q, Kc, Vc, [10], scale=json.load(open(GOLDEN))["scale"])
    return float(max(np.abs(a - b).max(), np.abs(c - d).max()))


def pin_shared_decode():
    """Shared-cache decode: the nq rows of each (slot, layer, head) equal the
    full-window matrix formula on that block of queries, and brute force."""
    B, nq, L, H, T, dh = 2, 5, 2, 2, 9, 64
    Q = _rand((B, nq, L, H, dh), 100)
    Kc, Vc = _rand((B, L, H, T, dh), 101), _rand((B, L, H, T, dh), 102)
    kl = np.array([9, 4])
    out = O.decode_shared(Q, Kc, Vc, kl)
    err = 0.0
    for b in range(B):
        for l in range(L):
            for h in range(H):
                full = O.full_window(Q[b, :, l, h], Kc[b, l, h], Vc[b, l, h], int(kl[b]), 0.125)
                err = max(err, float(np.abs(out[b, :, l, h] - full).max()))
                for n in (0, nq - 1):
                    bf = bf_attend(Q[b, n, l, h], Kc[b, l, h], Vc[b, l, h], int(kl[b]), 0.125)
                    err = max(err, float(np.abs(out[b, n, l, h] - np.array(bf)).max()))
    one = O.decode_shared(Q[:, :1], Kc, Vc, kl)[:, 0]
    err = max(err, float(np.abs(one - O.decode(Q[:, 0], Kc, Vc, kl)).max()))
    return err


def pin_populate_head():
    """One head's K/V block equals the head's slice of the whole projection, and
    pure-Python brute force, on shapes where every head is checked (the first
    and last column blocks, a bias on every column)."""
    err = 0.0
    for (B, T, d, L, H, dh) in [(2, 3, 4, 2, 2, 2), (1, 2, 6, 1, 3, 2), (1, 4, 8, 2, 2, 4)]:
        E, WK, WV = _rand((B, T, d), 160), _rand((L, d, d), 161), _rand((L, d, d), 162)
        bV = _rand((L, d), 163)
        Kb, Vb = bf_populate(E, WK, WV, bV, H)
        for b in range(B):
            for l in range(L):
                for h in range(H):
                    K, V = O.populate_head(E[b], WK[l], WV[l], bV[l], h, dh)
                    err = max(err, np.abs(K - Kb[b, l, h]).max(), np.abs(V - Vb[b, l, h]).max())
    B, T, d, L, H = 2, 37, 256, 2, 4
    E, WK, WV = _rand((B, T, d), 164), _rand((L, d, d), 165, d ** -0.5), _rand((L, d, d), 166, d ** -0.5)
    bV = _rand((L, d), 167, 0.02)
    Kc, Vc = O.populate(E, WK, WV, bV, H)
    for (b, l, h) in [(0, 0, 0), (1, 1, 3), (0, 1, 2), (1, 0, 1)]:
        K, V = O.populate_head(E[b], WK[l], WV[l], bV[l], h)
        err = max(err, np.abs(K - Kc[b, l, h]).max() / np.abs(Kc[b, l, h]).max(),
                  np.abs(V - Vc[b, l, h]).max() / np.abs(Vc[b, l, h]).max())
    return float(err)


def pin_rel_frobenius():
    """The populate error measure against ratios computed by hand:
    ||(8, -6)|| / ||(3, 4)|| = 10 / 5 = 2 (a perturbation orthogonal to the
    reference, so a missing square root gives 4 or 20 and a squared
    denominator 0.4); a 2x2 block with one element off by 3 over a reference of
    norm 5 gives 0.6; a uniform relative error eps gives eps; equality gives 0."""
    errs = [abs(O.rel_frobenius([11.0, -2.0], [3.0, 4.0]) - 2.0),
            abs(O.rel_frobenius([[1.0, 2.0], [2.0, 7.0]], [[1.0, 2.0], [2.0, 4.0]]) - 0.6)]
    ref = _rand((3, 5, 7), 170)
    errs.append(abs(O.rel_frobenius(ref * (1.0 + 3e-4), ref) - 3e-4) / 3e-4)
    errs.append(O.rel_frobenius(ref, ref))
    return float(max(errs))


def pin_round_bf16():
    """Hand-computed roundings (exact ties to even in both directions, just past
    a tie, negative values, the overflow threshold, subnormals: bf16's smallest
    spacing is 2^-133, so 1.5 * 2^-133 is a tie that goes to the even 2^-132 and
    2^-140 goes to 0), invariants
    (idempotent, low 16 bits clear, within half an ulp, monotonic) and agreement
    with the add-and-shift bit formulation of the same rule on 2^20 random
    patterns. Returns the number of failures."""
    u = 2.0 ** -8                                   # half an ulp of bf16 at 1.0
    cases = [(1.0, 1.0), (1.0 + u, 1.0), (1.0 + 3 * u, 1.0 + 4 * u), (1.0 + u + 2.0 ** -20, 1.0 + 2 * u),
             (-(1.0 + u + 2.0 ** -20), -(1.0 + 2 * u)), (-(1.0 + 3 * u), -(1.0 + 4 * u)), (0.0, 0.0),
             (float(np.finfo(np.float32).max), np.inf), (-float(np.finfo(np.float32).max), -np.inf),
             (1.5 * 2.0 ** -133, 2.0 ** -132), (1.25 * 2.0 ** -133, 2.0 ** -133), (2.0 ** -140, 0.0),
             (np.inf, np.inf)]
    bad = 0
    for x, want in cases:
        got = float(O.round_bf16(np.float32(x)))
        bad += int(got != want)
    bad += int(not np.isnan(O.round_bf16(np.float32(np.nan))))
    rng = np.random.default_rng(171)
    pat = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = pat.view(np.float32)
    x = x[np.isfinite(x)]
    r = O.round_bf16(x)
    bad += int((r.view(np.uint32) & np.uint32(0xFFFF)).any())
    fin = np.isfinite(r)
    bad += int(not np.array_equal(O.round_bf16(r[fin]), r[fin]))
    xs = np.sort(x[np.abs(x) < 1e30])
    bad += int((np.diff(O.round_bf16(xs).astype(np.float64)) < 0).any())
    ex = np.floor(np.log2(np.abs(xs[xs != 0].astype(np.float64))))
    half_ulp = 2.0 ** (np.maximum(ex, -126) - 8)
    bad += int((np.abs(O.round_bf16(xs[xs != 0]).astype(np.float64) - xs[xs != 0]) > half_ulp).any())
    bad += int(not np.array_equal(r.view(np.uint32) >> np.uint32(16), W.bf16_bits(x).astype(np.uint32)))
    return bad


def bf_layer_norm(x, gamma, beta, eps):
    x = list(x)
    d = len(x)
    mean = math.fsum(x) / d
    var = math.fsum((v - mean) ** 2 for v in x) / d
    return [(v - mean) / math.sqrt(var + eps) * g + b for v, g, b in zip(x, gamma, beta)]


def pin_cross_block():
    """LayerNorm closed forms; the block against a pure-Python restatement
    (fsum sums); WO = 0 leaves x unchanged; decode_layers equals decode on the
    layer slice."""
    errs = []
    # LayerNorm: constant row -> beta; normalised row has mean 0, variance 1
    errs.append(np.abs(O.layer_norm(np.full((1, 8), 3.0), np.ones(8), np.arange(8.0), 1e-5) - np.arange(8.0)).max())
    y = O.layer_norm(_rand((3, 64), 110), eps=0.0)
    errs.append(np.abs(y.mean(axis=1)).max())
    errs.append(np.abs(y.var(axis=1) - 1.0).max())
    B, L, H, T, dh = 2, 3, 2, 6, 64
    d = H * dh
    Kc, Vc = _rand((B, L, H, T, dh), 111), _rand((B, L, H, T, dh), 112)
    x = _rand((B, d), 113)
    WQ, WO = _rand((d, d), 114, d ** -0.5), _rand((d, d), 115, d ** -0.5)
    g, be, bQ, bO = _rand((d,), 116), _rand((d,), 117), _rand((d,), 118), _rand((d,), 119)
    kl = np.array([6, 4])
    out = O.cross_block(x, 1, Kc, Vc, kl, WQ, WO, g, be, 1e-5, bQ, bO)
    for b in range(B):
        hb = bf_layer_norm(x[b], g, be, 1e-5)
        q = [math.fsum(hb[i] * WQ[i][j] for i in range(d)) + bQ[j] for j in range(d)]
        a = []
        for h in range(H):
            a += bf_attend(q[h * dh:(h + 1) * dh], Kc[b, 1, h], Vc[b, 1, h], int(kl[b]), 0.125)
        ref = [x[b][j] + math.fsum(a[i] * WO[i][j] for i in range(d)) + bO[j] for j in range(d)]
        errs.append(np.abs(out[b] - np.array(ref)).max())
    errs.append(np.abs(O.cross_block(x, 2, Kc, Vc, kl, WQ, np.zeros((d, d))) - x).max())
    Ql = _rand((B, 2, H, dh), 120)
    errs.append(np.abs(O.decode_layers(Ql, Kc, Vc, kl, 1) - O.decode(Ql, Kc[:, 1:3], Vc[:, 1:3], kl)).max())
    return float(max(errs))


def pin_self_attention():
    """Token-by-token decode over a masked-blend cache equals the causal
    whole-window formula ("Recurrence as feeds": the two formulas match); the
    blend writes exactly one row and leaves the others."""
    errs = []
    for S, dh in ((1, 64), (2, 2), (7, 64), (20, 64)):
        Qs, Ks, Vs = _rand((S, dh), 130 + S), _rand((S, dh), 131 + S), _rand((S, dh), 132 + S)
        a = O.self_attention_steps(Qs, Ks, Vs)
        b = O.causal_full_window(Qs, Ks, Vs)
        errs.append(np.abs(a - b).max())
        errs.append(np.abs(a[0] - Vs[0]).max())            # the first token sees only itself
        if S >= 2:
            ref = bf_attend(Qs[1], Ks[:2], Vs[:2], 2, 1.0 / math.sqrt(dh))
            errs.append(np.abs(a[1] - np.array(ref)).max())
    c = _rand((5, 4), 140)
    u = O.masked_blend_update(c, np.full(4, 9.0), 3)
    errs.append(np.abs(np.delete(u, 3, axis=0) - np.delete(c, 3, axis=0)).max())
    errs.append(np.abs(u[3] - 9.0).max())
    errs.append(np.abs(O.masked_blend_update(c, np.full(4, 9.0), 5) - c).max())   # out of range: unchanged
    return float(max(errs))


def pin_attention_weights():
    """Each selected head's row sums to 1 over the valid keys and is zero beyond;
    weighting V by it gives the decode output of that head; brute force."""
    errs = []
    B, L, H, T, dh = 3, 2, 3, 9, 64
    Q, Kc, Vc = _rand((B, L, H, dh), 150), _rand((B, L, H, T, dh), 151), _rand((B, L, H, T, dh), 152)
    kl = np.array([9, 5, 0])
    heads = [(0, 2), (1, 0), (1, 2)]
    w, m = O.attention_weights(Q, Kc, kl, heads)
    dec = O.decode(Q, Kc, Vc, kl)
    for b in range(B):
        for k, (l, h) in enumerate(heads):
            n = int(kl[b])
            errs.append(abs(w[b, k].sum() - (1.0 if n > 0 else 0.0)))
            errs.append(np.abs(w[b, k, n:]).max() if n < T else 0.0)
            errs.append(np.abs(w[b, k] @ Vc[b, l, h] - dec[b, l, h]).max())
            if n > 0:
                e = [math.exp(0.125 * math.fsum(Q[b, l, h, c] * Kc[b, l, h, t, c] for c in range(dh))) for t in range(n)]
                z = math.fsum(e)
                errs.append(np.abs(w[b, k, :n] - np.array(e) / z).max())
    errs.append(np.abs(m - w.mean(axis=1)).max())
    return float(max(errs))


# ---------------------------------------------------------------------------
# the pins on the real oracle
# ---------------------------------------------------------------------------
def test_populate_matches_bruteforce():
    assert pin_populate_bruteforce() < 1e-12


def test_decode_matches_bruteforce():
    assert pin_decode_bruteforce() < 1e-12


def test_closed_forms():
    assert pin_closed_forms() < 1e-12


def test_key_bias_invariance():
    assert pin_key_bias_invariance() < 1e-12


def test_full_window_row():
    assert pin_full_window() < 1e-13


def test_cache_reuse_equals_reprojection():
    assert pin_cache_reuse() == 0.0


def test_layout_offset_whisper_base():
    assert pin_layout_offset() == 0


def test_token_major_cache_gives_a_different_answer():
    assert pin_token_major_rejected() > 1e-3


def test_scale_applies_to_scores():
    assert pin_scale_on_scores() < 1e-13


def test_shared_decode_matches_full_window_and_bruteforce():
    assert pin_shared_decode() < 1e-12


def test_cross_block_layer_norm_and_projections():
    assert pin_cross_block() < 1e-11


def test_self_attention_cache_matches_causal_window():
    assert pin_self_attention() < 1e-12


def test_alignment_head_weights():
    assert pin_attention_weights() < 1e-12


def test_populate_head_matches_projection_and_bruteforce():
    assert pin_populate_head() < 1e-12


def test_rel_frobenius_hand_computed():
    assert pin_rel_frobenius() < 1e-12


def test_round_bf16_hand_values_and_invariants():
    assert pin_round_bf16() == 0


def test_geometry_fails_closed():
    with pytest.raises(ValueError):
        O.populate(np.zeros((1, 0, 128)), np.zeros((1, 128, 128)), np.zeros((1, 128, 128)), np.zeros((1, 128)), 2)
    with pytest.raises(ValueError):
        O.check_geometry(10, 128, 3, 64)


def test_golden_call_arguments():
    g = json.load(open(GOLDEN))
    assert g["num_heads"] * g["head_dim"] == g["encoder_memory_shape"][1]
    assert g["scale"] == 1.0 / math.sqrt(g["head_dim"])
    assert g["key_tokens"] == g["encoder_memory_shape"][0]
    assert g["layer5_k_cache_offset_bytes"] == 5 * g["key_tokens"] * g["encoder_memory_shape"][1] * 4


def test_padding_rows_never_reach_the_output():
    B, L, H, T, dh = 2, 1, 2, 8, 64
    Q, Kc, Vc = _rand((B, L, H, dh), 90), _rand((B, L, H, T, dh), 91), _rand((B, L, H, T, dh), 92)
    ref = O.decode(Q, Kc, Vc, [5, 3])
    Kp, Vp = Kc.copy(), Vc.copy()
    Kp[0, :, :, 5:] = np.nan
    Vp[0, :, :, 5:] = np.inf
    Kp[1, :, :, 3:] = np.inf
    Vp[1, :, :, 3:] = np.nan
    assert np.array_equal(O.decode(Q, Kp, Vp, [5, 3]), ref)


# ---------------------------------------------------------------------------
# planted mistakes: each must make some pin fail
# ---------------------------------------------------------------------------
def _mut_transposed_w(monkeypatch):
    orig = O.populate

    def populate(E, WK, WV, bV, H, bK=None):
        return orig(E, np.swapaxes(np.asarray(WK, float), 1, 2), np.swapaxes(np.asarray(WV, float), 1, 2), bV, H, bK)
    monkeypatch.setattr(O, "populate", populate)


def _mut_interleaved_heads(monkeypatch):
    def head_major(X, H):
        T, d = X.shape
        return X.reshape(T, d // H, H).transpose(2, 0, 1).copy()
    monkeypatch.setattr(O, "head_major", head_major)


def _mut_token_major_slab(monkeypatch):
    def head_major(X, H):
        T, d = X.shape
        return X.reshape(H, T, d // H).copy()
    monkeypatch.setattr(O, "head_major", head_major)


def _mut_bias_on_keys(monkeypatch):
    orig = O.populate

    def populate(E, WK, WV, bV, H, bK=None):
        K, V = orig(E, WK, WV, np.zeros_like(np.asarray(bV, float)), H, bK)
        K2, _ = orig(E, WK, WV, np.zeros_like(np.asarray(bV, float)), H, bV)
        return K2, V
    monkeypatch.setattr(O, "populate", populate)


def _mut_sign_flip(monkeypatch):
    def attend_row(q, K, V, n, scale):
        return O.__dict__["_orig_attend"](q, K, V, n, -scale)
    monkeypatch.setitem(O.__dict__, "_orig_attend", O.attend_row)
    monkeypatch.setattr(O, "attend_row", attend_row)


def _mut_mask_off_by_one(monkeypatch):
    def attend_row(q, K, V, n, scale):
        return O.__dict__["_orig_attend"](q, K, V, n - 1, scale)
    monkeypatch.setitem(O.__dict__, "_orig_attend", O.attend_row)
    monkeypatch.setattr(O, "attend_row", attend_row)


def _mut_no_normalisation(monkeypatch):
    def attend_row(q, K, V, n, scale):
        q, K, V = np.asarray(q, float), np.asarray(K, float), np.asarray(V, float)
        if n <= 0:
            return np.zeros(q.shape[0])
        s = scale * (K[:n] @ q)
        w = np.exp(s - s.max())
        return w @ V[:n]
    monkeypatch.setattr(O, "attend_row", attend_row)


def _mut_missing_scale(monkeypatch):
    def attend_row(q, K, V, n, scale):
        return O.__dict__["_orig_attend"](q, K, V, n, 1.0)
    monkeypatch.setitem(O.__dict__, "_orig_attend", O.attend_row)
    monkeypatch.setattr(O, "attend_row", attend_row)


def _mut_head_without_bias(monkeypatch):
    orig = O.populate_head

    def populate_head(E_b, WK_l, WV_l, bV_l, h, dh=64):
        return orig(E_b, WK_l, WV_l, np.zeros_like(np.asarray(bV_l, float)), h, dh)
    monkeypatch.setattr(O, "populate_head", populate_head)


def _mut_head_neighbouring_block(monkeypatch):
    orig = O.populate_head

    def populate_head(E_b, WK_l, WV_l, bV_l, h, dh=64):
        return orig(E_b, WK_l, WV_l, bV_l, (h + 1) % (np.shape(WK_l)[1] // dh), dh)
    monkeypatch.setattr(O, "populate_head", populate_head)


def _mut_frobenius_without_sqrt(monkeypatch):
    def rel_frobenius(x, ref):
        x, ref = np.asarray(x, float), np.asarray(ref, float)
        return float(((x - ref) ** 2).sum() / max((ref ** 2).sum(), 1e-300))
    monkeypatch.setattr(O, "rel_frobenius", rel_frobenius)


def _mut_frobenius_squared_denominator(monkeypatch):
    def rel_frobenius(x, ref):
        x, ref = np.asarray(x, float), np.asarray(ref, float)
        return float(np.linalg.norm((x - ref).ravel()) / max((ref ** 2).sum(), 1e-300))
    monkeypatch.setattr(O, "rel_frobenius", rel_frobenius)


def _mut_round_half_away(monkeypatch):
    def round_bf16(x):
        u = np.array(x, dtype=np.float32).view(np.uint32)
        return ((u + np.uint32(0x8000)) & np.uint32(0xFFFF0000)).view(np.float32)
    monkeypatch.setattr(O, "round_bf16", round_bf16)


def _mut_round_truncate(monkeypatch):
    def round_bf16(x):
        u = np.array(x, dtype=np.float32).view(np.uint32)
        return (u & np.uint32(0xFFFF0000)).view(np.float32)
    monkeypatch.setattr(O, "round_bf16", round_bf16)


def _mut_layer_norm_unbiased(monkeypatch):
    def layer_norm(x, gamma=None, beta=None, eps=1e-5):
        x = np.asarray(x, np.float64)
        mean = x.mean(axis=-1, keepdims=True)
        var = ((x - mean) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)
        y = (x - mean) / np.sqrt(var + eps)
        return y * (1.0 if gamma is None else np.asarray(gamma)) + (0.0 if beta is None else np.asarray(beta))
    monkeypatch.setattr(O, "layer_norm", layer_norm)


def _mut_layer_norm_eps_outside_root(monkeypatch):
    def layer_norm(x, gamma=None, beta=None, eps=1e-5):
        x = np.asarray(x, np.float64)
        mean = x.mean(axis=-1, keepdims=True)
        y = (x - mean) / (np.sqrt(((x - mean) ** 2).mean(axis=-1, keepdims=True)) + eps)
        return y * (1.0 if gamma is None else np.asarray(gamma)) + (0.0 if beta is None else np.asarray(beta))
    monkeypatch.setattr(O, "layer_norm", layer_norm)


def _mut_block_without_residual(monkeypatch):
    orig = O.cross_block

    def cross_block(x, *args, **kw):
        return orig(x, *args, **kw) - np.asarray(x, np.float64)
    monkeypatch.setattr(O, "cross_block", cross_block)


def _mut_causal_window_excludes_self(monkeypatch):
    def self_attention_steps(Qs, Ks, Vs, scale=None):
        Qs, Ks, Vs = (np.asarray(a, np.float64) for a in (Qs, Ks, Vs))
        S, dh = Qs.shape
        scale = 1.0 / np.sqrt(dh) if scale is None else scale
        return np.stack([O.attend_row(Qs[i], Ks, Vs, i, scale) for i in range(S)])
    monkeypatch.setattr(O, "self_attention_steps", self_attention_steps)


def _mut_alignment_unmasked(monkeypatch):
    def attention_weights(Q, Kc, key_len, heads, scale=None):
        Q, Kc = np.asarray(Q, np.float64), np.asarray(Kc, np.float64)
        B, T = Kc.shape[0], Kc.shape[3]
        w = np.zeros((B, len(heads), T))
        for b in range(B):
            for k, (l, h) in enumerate(heads):
                s = 0.125 * (Kc[b, l, h] @ Q[b, l, h])
                e = np.exp(s - s.max())
                w[b, k] = e / e.sum()
        return w, w.mean(axis=1)
    monkeypatch.setattr(O, "attention_weights", attention_weights)


def _mut_alignment_mean_drops_a_head(monkeypatch):
    orig = O.attention_weights

    def attention_weights(*args, **kw):
        w, _ = orig(*args, **kw)
        return w, w[:, :-1].mean(axis=1)
    monkeypatch.setattr(O, "attention_weights", attention_weights)


def _mut_shared_decode_first_query(monkeypatch):
    orig = O.decode_shared

    def decode_shared(Q, Kc, Vc, key_len, scale=None):
        Q = np.asarray(Q, np.float64)
        return orig(np.repeat(Q[:, :1], Q.shape[1], axis=1), Kc, Vc, key_len, scale)
    monkeypatch.setattr(O, "decode_shared", decode_shared)


def _mut_decode_layers_next_layer(monkeypatch):
    def decode_layers(Q, Kc, Vc, key_len, l0, scale=None):
        Q = np.asarray(Q, np.float64)
        nl = Q.shape[1]
        return O.decode(Q, np.asarray(Kc)[:, l0 + 1:l0 + 1 + nl], np.asarray(Vc)[:, l0 + 1:l0 + 1 + nl], key_len,
                        scale)
    monkeypatch.setattr(O, "decode_layers", decode_layers)


def _mut_masked_blend_next_row(monkeypatch):
    def masked_blend_update(cache, new_row, pos):
        cache = np.asarray(cache, np.float64)
        mask = np.zeros((cache.shape[0], 1))
        if 0 <= pos + 1 < cache.shape[0]:
            mask[pos + 1, 0] = 1.0
        return cache * (1.0 - mask) + np.asarray(new_row, np.float64)[None, :] * mask
    monkeypatch.setattr(O, "masked_blend_update", masked_blend_update)


def _all_pins_pass():
    try:
        return (pin_populate_bruteforce() < 1e-12 and pin_decode_bruteforce() < 1e-12
                and pin_closed_forms() < 1e-12 and pin_full_window() < 1e-13 and pin_shared_decode() < 1e-12
                and pin_layout_offset() == 0 and pin_scale_on_scores() < 1e-13
                and pin_populate_head() < 1e-12 and pin_rel_frobenius() < 1e-12 and pin_round_bf16() == 0
                and pin_cross_block() < 1e-11 and pin_self_attention() < 1e-12
                and pin_attention_weights() < 1e-12)
    except (ValueError, IndexError, TypeError):   # a broken shape is a failed pin too
        return False


@pytest.mark.parametrize("mutation", [
    _mut_transposed_w, _mut_interleaved_heads, _mut_token_major_slab, _mut_bias_on_keys,
    _mut_sign_flip, _mut_mask_off_by_one, _mut_no_normalisation, _mut_missing_scale,
    _mut_head_without_bias, _mut_head_neighbouring_block, _mut_frobenius_without_sqrt,
    _mut_frobenius_squared_denominator, _mut_round_half_away, _mut_round_truncate,
    _mut_layer_norm_unbiased, _mut_layer_norm_eps_outside_root, _mut_block_without_residual,
    _mut_causal_window_excludes_self, _mut_alignment_unmasked, _mut_alignment_mean_drops_a_head,
    _mut_shared_decode_first_query, _mut_decode_layers_next_layer, _mut_masked_blend_next_row,
])
def test_planted_mistake_is_caught(monkeypatch, mutation):
    mutation(monkeypatch)
    assert not _all_pins_pass()
