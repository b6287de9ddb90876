"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Populate is compared element by element with the oracle's projection of the
same inputs: relative Frobenius over the cache, every element within the
arithmetic bound of TF32 / bf16 operands and the cache store, and every
(slot, layer, head) block's largest error against its largest value. Decode is
compared kernel-isolated -- the oracle decodes the very cache the GPU holds,
upcast to fp64 -- element by element (max-abs). Sizes span several tiles and
ragged tails; the full-size workloads are checked on sampled heads and rows.
"""
import numpy as np
import pytest
import torch

from _gpu_common import (DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, cache_for, check_populate, check_populate_head,
                         decode_policy, dev, host, inputs_on_device, populate_policy, record_parity)
from encoder_decoder_speech_gb300 import cxa
from encoder_decoder_speech_gb300 import workloads as W
from oracle import cross_attention as O

pytestmark = pytest.mark.gpu

DECODE_TOL = {"f32": DECODE_F32_MAX_ABS, "bf16": DECODE_BF16_MAX_ABS}


@pytest.fixture(scope="module", autouse=True)
def _lib(cxa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.synchronize()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def _populate(w, cache_dtype):
    d, h = inputs_on_device(w)
    c = cache_for(w, cache_dtype)
    c.populate(d["E"], d["WK"], d["WV"], d["bV"])
    torch.cuda.synchronize()
    return c, d, h


SMALL = [
    # name, B, T, d, L, H: tiles of 128 rows x 256 columns, ragged in both
    ("one_row", 1, 1, 64, 1, 1),
    ("two_mtiles_ragged", 2, 200, 128, 2, 2),
    ("three_ntiles", 3, 129, 384, 1, 6),
    ("odd_heads_straddle", 2, 300, 192, 3, 3),
    ("exact_tiles", 1, 256, 256, 2, 4),
]


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL, ids=[s[0] for s in SMALL])
def test_populate_small(shape, in_dtype, cache_dtype):
    name, B, T, d, L, H = shape
    w = W.custom(name, B=B, T=T, d=d, L=L, H=H, in_dtype=in_dtype, index=910)
    c, _, h = _populate(w, cache_dtype)
    check_populate(host(c.Kc), host(c.Vc), h["E"], h["WK"], h["WV"], h["bV"], H, in_dtype, cache_dtype, name)
    assert np.isfinite(host(c.Kc)).all() and np.isfinite(host(c.Vc)).all()


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_populate_tiny_config(cache_dtype):
    w = W.WORKLOADS["tiny"]
    c, _, h = _populate(w, cache_dtype)
    ek, ev, blk = check_populate(host(c.Kc), host(c.Vc), h["E"], h["WK"], h["WV"], h["bV"], w.H, "f32", cache_dtype,
                                 "tiny")
    print(f"tiny populate rel-frob K {ek:.3e} V {ev:.3e}, worst block {blk:.3e} ({cache_dtype} cache)")
    record_parity("tiny", f"{cache_dtype} cache", populate_rel_frob_K=ek, populate_rel_frob_V=ev,
                  populate_worst_block_ratio=blk)


def test_populate_partial_slots_leave_others_untouched():
    w = W.custom("partial", B=4, T=150, d=128, L=2, H=2, index=911)
    d, h = inputs_on_device(w)
    c = cache_for(w, "f32")
    c.Kc.fill_(7.0)
    c.Vc.fill_(7.0)
    c.populate(d["E"][1:3].contiguous(), d["WK"], d["WV"], d["bV"], b0=1)
    torch.cuda.synchronize()
    assert [c.is_ready(b) for b in range(4)] == [False, True, True, False]
    assert torch.all(c.Kc[0] == 7.0) and torch.all(c.Kc[3] == 7.0) and torch.all(c.Vc[3] == 7.0)
    check_populate(host(c.Kc[1:3]), host(c.Vc[1:3]), h["E"][1:3], h["WK"], h["WV"], h["bV"], w.H, "f32", "f32",
                   "partial")


def _fill_cache(c, seed):
    """Overwrite a populated cache with seeded N(0,1) values (bf16-exact for a bf16 cache)."""
    rng = np.random.default_rng(seed)
    K = rng.standard_normal(tuple(c.Kc.shape), dtype=np.float32)
    V = rng.standard_normal(tuple(c.Vc.shape), dtype=np.float32)
    if c.cache_dtype == "bf16":
        K, V = W.bf16_round(K), W.bf16_round(V)
    c.Kc.copy_(dev(K, c.Kc.dtype))
    c.Vc.copy_(dev(V, c.Vc.dtype))
    return K.astype(np.float64), V.astype(np.float64)


def _decode_case(T, key_len, cache_dtype, L=2, H=3, seed=0, scale=0.0):
    B = len(key_len)
    w = W.custom(f"dec{T}", B=B, T=T, d=64 * H, L=L, H=H, index=920)
    c, d, _ = _populate(w, cache_dtype)
    K, V = _fill_cache(c, 100 + seed)
    Q = np.random.default_rng(200 + seed).standard_normal((B, L, H, 64)).astype(np.float32)
    kl = np.array(key_len, dtype=np.int32)
    out = c.decode(dev(Q), dev(kl, torch.int32), scale=scale)
    torch.cuda.synchronize()
    ref = O.decode(Q, K, V, kl, scale if scale > 0 else None)
    return host(out), ref


DECODE_CASES = [
    (1, [1, 0]),
    (2, [2, 1, 0]),
    (3, [3, 2, 5, -4]),
    (63, [63, 1, 62]),
    (64, [64, 63, 1]),
    (65, [65, 64, 33]),
    (127, [127, 64, 65, 0]),
    (129, [129, 128, 100]),
    (1500, [1500, 500, 1, 1499, 2000]),
]


@pytest.mark.parametrize("shape", ["stream", "rows"])
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,key_len", DECODE_CASES, ids=[f"T{c[0]}" for c in DECODE_CASES])
def test_decode_kernel_isolated(T, key_len, cache_dtype, shape):
    with decode_policy(shape):
        got, ref = _decode_case(T, key_len, cache_dtype, seed=T)
    err = np.abs(got - ref).max()
    assert err <= DECODE_TOL[cache_dtype], err
    for b, n in enumerate(key_len):
        if n <= 0:
            assert np.all(got[b] == 0.0)


def test_decode_scale_override():
    got, ref = _decode_case(300, [300, 150], "f32", scale=0.37, seed=3)
    assert np.abs(got - ref).max() <= DECODE_F32_MAX_ABS


def test_decode_repeated_calls_share_the_workspace():
    """The arrival counters are reset by each call: consecutive steps stay exact."""
    w = W.custom("rep", B=3, T=700, d=256, L=2, H=4, ragged=True, index=921)
    c, d, _ = _populate(w, "f32")
    K, V = host(c.Kc), host(c.Vc)
    kl = W.make_key_len(w)
    for s in range(4):
        Q = W.make_Q(w, s)
        out = host(c.decode(dev(Q), d["key_len"]))
        assert np.abs(out - O.decode(Q, K, V, kl)).max() <= DECODE_F32_MAX_ABS


@pytest.mark.parametrize("shape", ["stream", "rows"])
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_padding_rows_are_never_read(cache_dtype, shape):
    """NaN / Inf in cache rows t >= key_len[b] must not reach the output."""
    w = W.custom("poison", B=3, T=500, d=128, L=2, H=2, ragged=True, index=922)
    c, d, _ = _populate(w, cache_dtype)
    Q = dev(W.make_Q(w, 0))
    kl = W.make_key_len(w)
    with decode_policy(shape):
        clean = c.decode(Q, d["key_len"]).clone()
        for b in range(w.B):
            c.Kc[b, :, :, int(kl[b]):] = float("nan")
            c.Vc[b, :, :, int(kl[b]):] = float("inf")
        poisoned = c.decode(Q, d["key_len"])
        torch.cuda.synchronize()
    assert torch.equal(clean, poisoned)


def test_workspace_poison_does_not_leak():
    """Partials are fully rewritten each call: NaN-filled partial storage is harmless."""
    w = W.custom("wspoison", B=2, T=400, d=128, L=1, H=2, index=923)
    c, d, h = _populate(w, "f32")
    nctr = ((w.B * w.L * w.H * 4 + 255) // 256) * 256
    c.decode_ws[nctr:c.decode_ws_bytes].view(torch.float32).fill_(float("nan"))
    Q = W.make_Q(w, 0)
    out = host(c.decode(dev(Q), d["key_len"]))
    assert np.abs(out - O.decode(Q, host(c.Kc), host(c.Vc), h["key_len"])).max() <= DECODE_F32_MAX_ABS


def test_invalidate_refuses_then_repopulate():
    w = W.custom("inval", B=3, T=260, d=128, L=2, H=2, index=924)
    c, d, h = _populate(w, "f32")
    Q = dev(W.make_Q(w, 0))
    ref = c.decode(Q, d["key_len"]).clone()
    c.invalidate(1)
    out = torch.full_like(ref, 123.0)
    launches = cxa.cxa_launch_count()
    rc = cxa.cxa_decode(c.handle, Q, d["key_len"], out, 0.0, c.decode_ws, c.decode_ws_bytes)
    assert rc == cxa.CXA_ENOTREADY
    assert cxa.cxa_launch_count() == launches
    torch.cuda.synchronize()
    assert torch.all(out == 123.0)
    c.populate(d["E"][1:2].contiguous(), d["WK"], d["WV"], d["bV"], b0=1)
    again = c.decode(Q, d["key_len"])
    torch.cuda.synchronize()
    assert torch.allclose(again, ref, atol=1e-6, rtol=0)


def test_key_bias_folded_into_the_cache_leaves_decode_unchanged():
    """A key bias adds q.bK to every score of a row: softmax ignores it."""
    w = W.custom("kbias", B=2, T=333, d=256, L=2, H=4, index=925)
    c, d, _ = _populate(w, "f32")
    Q = dev(W.make_Q(w, 1))
    ref = c.decode(Q, d["key_len"]).clone()
    bK = dev(np.random.default_rng(5).standard_normal((w.L, w.H, 64)).astype(np.float32))
    c.Kc += bK[None, :, :, None, :]
    got = c.decode(Q, d["key_len"])
    torch.cuda.synchronize()
    assert (got - ref).abs().max().item() <= DECODE_F32_MAX_ABS


def test_whisper_base_layer5_slab_offset():
    """Whisper-Base dims, fp32 cache: the layer-5 K slab starts 15,360,000 bytes
    into slot 0 and holds K_5 = E x WK_5 head-major."""
    w = W.WORKLOADS["base"]
    c, _, h = _populate(w, "f32")
    flat = c.Kc.view(-1)
    off = 15360000 // 4
    got = host(flat[off:off + 64])
    ref = h["E"][0, 0].astype(np.float64) @ h["WK"][5][:, :64].astype(np.float64)
    assert np.abs(got - ref).max() <= 2e-3 * np.abs(ref).max()
    # token-major placement would put E[0, 1] x WK_5[:, 0] at offset + 512 instead
    ref_t1 = h["E"][0, 1].astype(np.float64) @ h["WK"][5][:, 0].astype(np.float64)
    assert abs(host(flat[off + 64:off + 65])[0] - ref_t1) <= 2e-3 * abs(ref_t1) + 1e-3


@pytest.mark.parametrize("name", ["tiny", "base"])
def test_config_end_to_end(name):
    """Full Tiny / Base workloads: populate parity, then every decode step
    kernel-isolated and end to end against the oracle from E."""
    w = W.WORKLOADS[name]
    c, d, h = _populate(w, "f32")
    Kg, Vg = host(c.Kc), host(c.Vc)
    ek, ev, blk = check_populate(Kg, Vg, h["E"], h["WK"], h["WV"], h["bV"], w.H, "f32", "f32", name)
    Kr, Vr = O.populate(h["E"], h["WK"], h["WV"], h["bV"], w.H)
    worst_iso = worst_e2e = 0.0
    for s in range(w.steps):
        Q = W.make_Q(w, s)
        out = host(c.decode(dev(Q), d["key_len"]))
        worst_iso = max(worst_iso, np.abs(out - O.decode(Q, Kg, Vg, h["key_len"])).max())
        if s < 4:
            worst_e2e = max(worst_e2e, np.abs(out - O.decode(Q, Kr, Vr, h["key_len"])).max())
    print(f"{name}: decode max-abs kernel-isolated {worst_iso:.2e}, end-to-end {worst_e2e:.2e}")
    record_parity(name, "f32 cache", populate_rel_frob_K=ek, populate_rel_frob_V=ev, populate_worst_block_ratio=blk,
                  decode_max_abs_kernel_isolated=worst_iso, decode_max_abs_end_to_end=worst_e2e,
                  decode_steps_checked=w.steps)
    assert worst_iso <= DECODE_F32_MAX_ABS


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_batched_base(cache_dtype):
    """Batched Whisper-Base (16 memories, ragged key_len): populate parity on every
    slot (element-wise and per head block), and every row of four decode steps
    both kernel-isolated (the oracle on the GPU's cache) and end to end (the
    oracle's own cache from E); the end-to-end error is gated for the bf16 cache
    and reported for the fp32 one."""
    w = W.WORKLOADS["batched_base"]
    c, d, h = _populate(w, cache_dtype)
    steps = (0, 1, 64, 127)
    Qs = {s: W.make_Q(w, s) for s in steps}
    outs = {s: host(c.decode(dev(Qs[s]), d["key_len"])) for s in steps}
    kl = h["key_len"]
    worst_iso = worst_e2e = worst_blk = worst_frob = 0.0
    for b in range(w.B):
        Kg, Vg = host(c.Kc[b:b + 1]), host(c.Vc[b:b + 1])
        fk, fv, blk = check_populate(Kg, Vg, h["E"][b:b + 1], h["WK"], h["WV"], h["bV"], w.H, "f32", cache_dtype,
                                     f"batched slot {b}")
        worst_blk = max(worst_blk, blk)
        worst_frob = max(worst_frob, fk, fv)
        Kr, Vr = O.populate(h["E"][b:b + 1], h["WK"], h["WV"], h["bV"], w.H)
        for s in steps:
            iso = O.decode(Qs[s][b:b + 1], Kg, Vg, kl[b:b + 1])
            e2e = O.decode(Qs[s][b:b + 1], Kr, Vr, kl[b:b + 1])
            worst_iso = max(worst_iso, float(np.abs(outs[s][b:b + 1] - iso).max()))
            worst_e2e = max(worst_e2e, float(np.abs(outs[s][b:b + 1] - e2e).max()))
    print(f"batched base ({cache_dtype} cache): worst populate block {worst_blk:.3e}, decode max-abs "
          f"kernel-isolated {worst_iso:.2e}, end-to-end {worst_e2e:.2e}")
    record_parity("batched_base", f"{cache_dtype} cache", populate_worst_slot_rel_frob=worst_frob,
                  populate_worst_block_ratio=worst_blk, decode_max_abs_kernel_isolated=worst_iso,
                  decode_max_abs_end_to_end=worst_e2e, slots=w.B, decode_steps_checked=len(steps))
    assert worst_iso <= DECODE_TOL[cache_dtype]
    if cache_dtype == "bf16":
        assert worst_e2e <= DECODE_BF16_MAX_ABS


def test_large_sampled_heads():
    """Whisper-large dims, bf16 inputs and cache, 8 memories: 48 sampled (slot,
    layer, head) K/V blocks (plus the first and last) against the oracle, element
    by element, and their decode rows both kernel-isolated and end to end."""
    w = W.WORKLOADS["large"]
    c, d, h = _populate(w, "bf16")
    rng = np.random.default_rng(77)
    heads = sorted({(int(rng.integers(w.B)), int(rng.integers(w.L)), int(rng.integers(w.H))) for _ in range(48)}
                   | {(0, 0, 0), (w.B - 1, w.L - 1, w.H - 1)})
    Q = W.make_Q(w, 0)
    out = host(c.decode(dev(Q), d["key_len"]))
    worst = dict(frob=0.0, blk=0.0, iso=0.0, e2e=0.0)
    for (b, l, hh) in heads:
        Kg, Vg = host(c.Kc[b, l, hh]), host(c.Vc[b, l, hh])
        fk, fv, blk, Kr, Vr = check_populate_head(Kg, Vg, h["E"][b], h["WK"][l], h["WV"][l], h["bV"][l], hh, "bf16",
                                                  "bf16", f"large ({b}, {l}, {hh})")
        iso = O.attend_row(Q[b, l, hh], Kg, Vg, w.T, w.scale)
        e2e = O.attend_row(Q[b, l, hh], Kr, Vr, w.T, w.scale)
        worst = dict(frob=max(worst["frob"], fk, fv), blk=max(worst["blk"], blk),
                     iso=max(worst["iso"], np.abs(out[b, l, hh] - iso).max()),
                     e2e=max(worst["e2e"], np.abs(out[b, l, hh] - e2e).max()))
        assert np.abs(out[b, l, hh] - iso).max() <= DECODE_BF16_MAX_ABS
        assert np.abs(out[b, l, hh] - e2e).max() <= DECODE_BF16_MAX_ABS
    record_parity("large", "bf16 inputs, bf16 cache", sampled_heads=len(heads), populate_worst_rel_frob=worst["frob"],
                  populate_worst_block_ratio=worst["blk"], decode_max_abs_kernel_isolated=worst["iso"],
                  decode_max_abs_end_to_end=worst["e2e"])


def test_large_dims_tf32_sampled_heads():
    """Whisper-large widths with fp32 inputs (TF32 operands, 40 k-blocks per tile,
    320 column tiles: the CTA-pair GEMM) into an fp32 cache, two memories: 24
    sampled (slot, layer, head) blocks element by element, and their decode rows."""
    w = W.custom("large_tf32", B=2, T=1500, d=1280, L=32, H=20, ragged=True, index=945)
    c, d, h = _populate(w, "f32")
    rng = np.random.default_rng(78)
    heads = sorted({(int(rng.integers(w.B)), int(rng.integers(w.L)), int(rng.integers(w.H))) for _ in range(24)}
                   | {(0, 0, 0), (w.B - 1, w.L - 1, w.H - 1)})
    Q = W.make_Q(w, 0)
    out = host(c.decode(dev(Q), d["key_len"]))
    for (b, l, hh) in heads:
        Kg, Vg = host(c.Kc[b, l, hh]), host(c.Vc[b, l, hh])
        check_populate_head(Kg, Vg, h["E"][b], h["WK"][l], h["WV"][l], h["bV"][l], hh, "f32", "f32",
                            f"large tf32 ({b}, {l}, {hh})")
        n = int(min(max(h["key_len"][b], 0), w.T))
        iso = O.attend_row(Q[b, l, hh], Kg, Vg, n, 0.125)
        assert np.abs(out[b, l, hh] - iso).max() <= DECODE_F32_MAX_ABS


@pytest.mark.parametrize("shape", ["stream", "rows", "alternate"])
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
def test_back_to_back_steps_without_sync(cache_dtype, shape):
    """Consecutive decode launches on one stream overlap (the next grid starts
    streaming the cache while the previous one finishes); every step's output
    must still be exact, with either kernel shape or the two alternating."""
    w = W.custom("b2b", B=5, T=900, d=384, L=2, H=6, ragged=True, index=926)
    c, d, h = _populate(w, cache_dtype)
    Kg, Vg = host(c.Kc), host(c.Vc)
    Qs = [W.make_Q(w, s) for s in range(12)]
    Qd = [dev(q) for q in Qs]
    outs = [torch.empty_like(Qd[0]) for _ in Qs]
    torch.cuda.synchronize()
    for i, (q, o) in enumerate(zip(Qd, outs)):
        pick = shape if shape != "alternate" else ("stream", "rows")[i % 2]
        with decode_policy(pick):
            c.decode(q, d["key_len"], out=o)
    torch.cuda.synchronize()
    for q, o in zip(Qs, outs):
        assert np.abs(host(o) - O.decode(q, Kg, Vg, h["key_len"])).max() <= DECODE_TOL[cache_dtype]


@pytest.mark.parametrize("shape", ["stream", "rows", "alternate"])
def test_chained_queries_read_after_the_previous_step(shape):
    """Step k+1's query buffer is step k's output buffer: the next launch must
    not read Q before the previous grid has written it."""
    w = W.custom("chain", B=3, T=1100, d=256, L=2, H=4, ragged=True, index=927)
    c, d, h = _populate(w, "f32")
    Kg, Vg = host(c.Kc), host(c.Vc)
    q0 = W.make_Q(w, 0)
    bufs = [dev(q0), torch.empty_like(dev(q0))]
    torch.cuda.synchronize()
    for k in range(10):
        pick = shape if shape != "alternate" else ("stream", "rows")[k % 2]
        with decode_policy(pick):
            c.decode(bufs[k % 2], d["key_len"], out=bufs[(k + 1) % 2])
    torch.cuda.synchronize()
    ref = q0.astype(np.float64)
    for k in range(10):
        ref = O.decode(ref, Kg, Vg, h["key_len"])
    assert np.abs(host(bufs[10 % 2]) - ref).max() <= DECODE_F32_MAX_ABS


def test_two_caches_interleaved_back_to_back():
    """Decodes of two caches (own workspaces) alternate on one stream without syncs."""
    w1 = W.custom("il1", B=2, T=640, d=128, L=3, H=2, ragged=True, index=928)
    w2 = W.custom("il2", B=4, T=333, d=256, L=1, H=4, index=929)
    c1, d1, h1 = _populate(w1, "f32")
    c2, d2, h2 = _populate(w2, "bf16")
    Q1 = [W.make_Q(w1, s) for s in range(6)]
    Q2 = [W.make_Q(w2, s) for s in range(6)]
    o1 = [torch.empty(q.shape, device="cuda") for q in Q1]
    o2 = [torch.empty(q.shape, device="cuda") for q in Q2]
    q1d, q2d = [dev(q) for q in Q1], [dev(q) for q in Q2]
    torch.cuda.synchronize()
    for s in range(6):
        c1.decode(q1d[s], d1["key_len"], out=o1[s])
        c2.decode(q2d[s], d2["key_len"], out=o2[s])
    torch.cuda.synchronize()
    for s in range(6):
        assert np.abs(host(o1[s]) - O.decode(Q1[s], host(c1.Kc), host(c1.Vc), h1["key_len"])).max() <= DECODE_F32_MAX_ABS
        assert np.abs(host(o2[s]) - O.decode(Q2[s], host(c2.Kc), host(c2.Vc), h2["key_len"])).max() <= DECODE_BF16_MAX_ABS


@pytest.mark.parametrize("in_dtype,cache_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f32", "bf16")])
def test_populate_from_weights_packed_once(in_dtype, cache_dtype):
    """Weights packed once (cxa_pack_weights) then several windows populated from
    the packed copy (cxa_populate_packed) give exactly the cache cxa_populate
    writes, and pass the oracle gates."""
    w = W.custom("packed", B=3, T=700, d=256, L=3, H=4, ragged=True, in_dtype=in_dtype, index=940)
    d, h = inputs_on_device(w)
    a = cache_for(w, cache_dtype)
    b = cache_for(w, cache_dtype)
    packed = b.pack_weights(d["WK"], d["WV"])
    for window in range(2):
        E = d["E"] if window == 0 else d["E"].flip(0).contiguous()
        Eh = h["E"] if window == 0 else h["E"][::-1].copy()
        a.populate(E, d["WK"], d["WV"], d["bV"])
        b.populate_packed(E, packed, d["bV"])
        torch.cuda.synchronize()
        assert all(b.is_ready(s) for s in range(w.B))
        assert torch.equal(a.Kc, b.Kc) and torch.equal(a.Vc, b.Vc)
        check_populate(host(b.Kc), host(b.Vc), Eh, h["WK"], h["WV"], h["bV"], w.H, in_dtype, cache_dtype,
                       f"packed window {window}")


# (name, B, T, d, L, H, input dtype, cache dtype) for the two GEMM shapes
POP_SHAPE_GEOMS = [
    ("ragged_T", 3, 700, 256, 2, 4, "f32", "f32"),      # T not a multiple of the pair's 256-row tile
    ("short_T", 2, 100, 128, 3, 2, "bf16", "bf16"),     # T <= 128: the odd CTA's rows all lie past T
    ("half_n_tile", 2, 333, 192, 3, 3, "f32", "bf16"),  # 18 heads: the last 256-column tile is half empty
    ("bf16_in_f32_cache", 3, 520, 128, 2, 2, "bf16", "f32"),  # the fourth dtype combination
]


@pytest.mark.parametrize("geom", POP_SHAPE_GEOMS, ids=[g[0] for g in POP_SHAPE_GEOMS])
def test_populate_pair_and_single_shapes_agree(geom):
    """The CTA-pair GEMM (cta_group::2, forced with CXA_POPULATE_PAIR, which fails
    rather than fall back) and the one-CTA GEMM write bit-identical caches that
    pass the oracle gates, on edges of the pair's 256 x 256 tile."""
    name, B, T, dm, L, H, in_dtype, cache_dtype = geom
    w = W.custom(name, B=B, T=T, d=dm, L=L, H=H, ragged=True, in_dtype=in_dtype, index=942)
    d, h = inputs_on_device(w)
    caches = {}
    for shape in ("single", "pair"):
        c = cache_for(w, cache_dtype)
        packed = c.pack_weights(d["WK"], d["WV"])
        with populate_policy(shape):
            c.populate_packed(d["E"], packed, d["bV"])
        torch.cuda.synchronize()
        caches[shape] = c
    assert torch.equal(caches["single"].Kc, caches["pair"].Kc)
    assert torch.equal(caches["single"].Vc, caches["pair"].Vc)
    check_populate(host(caches["pair"].Kc), host(caches["pair"].Vc), h["E"], h["WK"], h["WV"], h["bV"], w.H,
                   in_dtype, cache_dtype, name)
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def test_populate_pair_partial_slots():
    """A populate of slots [1, 3) of a 4-slot cache on CTA pairs writes those slots
    exactly as one CTA per tile does and leaves slots 0 and 3 as they were."""
    w = W.custom("pair_partial", B=4, T=600, d=256, L=2, H=4, ragged=True, index=943)
    d, h = inputs_on_device(w)
    E = d["E"][1:3].contiguous()
    out = {}
    for shape in ("single", "pair"):
        c = cache_for(w, "f32")
        c.Kc.fill_(7.0)
        c.Vc.fill_(-7.0)
        packed = c.pack_weights(d["WK"], d["WV"])
        with populate_policy(shape):
            c.populate_packed(E, packed, d["bV"], b0=1)
        torch.cuda.synchronize()
        assert [c.is_ready(b) for b in range(w.B)] == [False, True, True, False]
        for b in (0, 3):
            assert bool((c.Kc[b] == 7.0).all()) and bool((c.Vc[b] == -7.0).all())
        out[shape] = c
    assert torch.equal(out["single"].Kc, out["pair"].Kc) and torch.equal(out["single"].Vc, out["pair"].Vc)
    check_populate(host(out["pair"].Kc[1:3]), host(out["pair"].Vc[1:3]), h["E"][1:3], h["WK"], h["WV"], h["bV"],
                   w.H, "f32", "f32", "pair partial")


def test_populate_packed_refuses_a_short_buffer():
    w = W.custom("packed_short", B=1, T=64, d=128, L=2, H=2, index=941)
    d, _ = inputs_on_device(w)
    c = cache_for(w, "f32")
    packed = c.pack_weights(d["WK"], d["WV"])
    launches = cxa.cxa_launch_count()
    rc = cxa.cxa_populate_packed(c.handle, 0, 1, d["E"], packed, packed.numel() - 16, d["bV"], w.T, w.d, w.L, w.H,
                                 cxa.CXA_F32)
    assert rc == cxa.CXA_EINVAL and cxa.cxa_launch_count() == launches
    assert not c.is_ready(0)
