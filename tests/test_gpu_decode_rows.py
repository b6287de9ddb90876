"""The latency shape of the one-query decode (a cluster of C CTAs per (slot,
layer, head) row, C the largest size up to 8 whose clusters are all resident)
against the oracle, kernel-isolated: 1 to 300 rows, which take clusters of 8
down to 1 CTA and both warp counts; rows long enough that every warp refills its
ring many times; key lengths 0, 1, fewer keys than CTAs in
the cluster, share boundaries inside a sub-chunk, the whole cache, beyond T and
negative; both cache dtypes; a layer range; and the automatic choice, which
must take the stream kernel once the rows no longer fit or the stream is long,
with unchanged results."""
import numpy as np
import pytest
import torch

from _gpu_common import DECODE_BF16_MAX_ABS, DECODE_F32_MAX_ABS, cache_for, decode_policy, dev, host
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
    cxa.cxa_set_decode_policy(cxa.CXA_DECODE_AUTO)
    assert cxa.cxa_device_status(1) == cxa.CXA_OK


def _filled(B, T, L, H, cache_dtype, seed):
    """A cache of seeded N(0,1) rows (bf16-exact for a bf16 cache), marked ready
    through a populate of zero weights first."""
    w = W.custom("rowsfill", B=B, T=T, d=64 * H, L=L, H=H, index=950)
    c = cache_for(w, cache_dtype)
    E = torch.zeros((B, T, 64 * H), device="cuda")
    Wz = torch.zeros((L, 64 * H, 64 * H), device="cuda")
    c.populate(E, Wz, Wz, torch.zeros((L, 64 * H), device="cuda"))
    rng = np.random.default_rng(seed)
    K = rng.standard_normal(tuple(c.Kc.shape), dtype=np.float32)
    V = rng.standard_normal(tuple(c.Vc.shape), dtype=np.float32)
    if cache_dtype == "bf16":
        K, V = W.bf16_round(K), W.bf16_round(V)
    c.Kc.copy_(dev(K, c.Kc.dtype))
    c.Vc.copy_(dev(V, c.Vc.dtype))
    return c, K.astype(np.float64), V.astype(np.float64)


# (B, L, H) -> rows = B*L*H from 1 to 300 (cluster sizes 8 down to 1)
GEOMS = [(1, 1, 1), (2, 2, 6), (2, 19, 1), (1, 6, 8), (3, 4, 5), (2, 2, 19), (5, 4, 5), (7, 4, 5), (5, 5, 8),
         (5, 6, 10)]


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("geom", GEOMS, ids=[f"rows{g[0] * g[1] * g[2]}" for g in GEOMS])
def test_rows_kernel_every_cluster_size(geom, cache_dtype):
    B, L, H = geom
    T = 1500
    c, K, V = _filled(B, T, L, H, cache_dtype, seed=B * 100 + L * 10 + H)
    rng = np.random.default_rng(7)
    choices = [0, 1, 3, 7, 31, 33, 65, 700, 1499, 1500, 1700, -2]
    kl = np.array([choices[(i * 5 + 3) % len(choices)] if i else 1500 for i in range(B)], dtype=np.int32)
    kl[rng.integers(B)] = choices[int(rng.integers(len(choices)))]
    Q = rng.standard_normal((B, L, H, 64)).astype(np.float32)
    with decode_policy("rows"):
        out = host(c.decode(dev(Q), dev(kl, torch.int32)))
    ref = O.decode(Q, K, V, kl)
    assert np.abs(out - ref).max() <= TOL[cache_dtype]
    for b in range(B):
        if kl[b] <= 0:
            assert np.all(out[b] == 0.0)


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 31, 32, 33, 64, 257])
def test_rows_kernel_short_memories(T, cache_dtype):
    """Every key length of a short memory, one slot per key length."""
    B, L, H = T + 1 if T < 40 else 12, 1, 2
    c, K, V = _filled(B, T, L, H, cache_dtype, seed=T)
    kl = np.array([min(b * max(1, T // 10), T) for b in range(B)], dtype=np.int32)
    Q = np.random.default_rng(T).standard_normal((B, L, H, 64)).astype(np.float32)
    with decode_policy("rows"):
        out = host(c.decode(dev(Q), dev(kl, torch.int32)))
    assert np.abs(out - O.decode(Q, K, V, kl)).max() <= TOL[cache_dtype]


def test_rows_kernel_layer_range():
    B, L, H, T = 2, 6, 8, 1500
    c, K, V = _filled(B, T, L, H, "f32", seed=3)
    kl = np.array([1500, 777], dtype=np.int32)
    Q = np.random.default_rng(3).standard_normal((B, 2, H, 64)).astype(np.float32)
    out = torch.empty((B, 2, H, 64), device="cuda")
    with decode_policy("rows"):
        c.decode_layers(3, dev(Q), dev(kl, torch.int32), out=out)
    ref = O.decode_layers(Q, K, V, kl, 3)
    assert np.abs(host(out) - ref).max() <= DECODE_F32_MAX_ABS


@pytest.mark.parametrize("geom", [(4, 6, 8), (1, 6, 8), (1, 6, 8, 8192)])
def test_automatic_choice_gives_the_same_result(geom):
    """192 rows (do not fit: stream kernel), 48 rows of 1500 keys (latency shape),
    48 rows of 8192 keys (a long stream: stream kernel) -- all equal the oracle
    and agree with the forced stream kernel."""
    B, L, H = geom[:3]
    T = geom[3] if len(geom) > 3 else 1500
    c, K, V = _filled(B, T, L, H, "f32", seed=11)
    kl = np.full(B, T, dtype=np.int32)
    Q = np.random.default_rng(11).standard_normal((B, L, H, 64)).astype(np.float32)
    with decode_policy("auto"):
        a = host(c.decode(dev(Q), dev(kl, torch.int32)))
    with decode_policy("stream"):
        s = host(c.decode(dev(Q), dev(kl, torch.int32)))
    ref = O.decode(Q, K, V, kl)
    assert np.abs(a - ref).max() <= DECODE_F32_MAX_ABS
    assert np.abs(s - ref).max() <= DECODE_F32_MAX_ABS


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [3000, 8192])
def test_rows_kernel_long_rows_refill_the_rings(T, cache_dtype):
    """A single memory of 3000 or 8192 keys forced onto the latency shape: each warp
    works through many sub-chunks, refilling its two stages, and the result agrees
    with the oracle."""
    B, L, H = 1, 6, 8
    c, K, V = _filled(B, T, L, H, cache_dtype, seed=T + 1)
    kl = np.array([T - 37], dtype=np.int32)
    Q = np.random.default_rng(T).standard_normal((B, L, H, 64)).astype(np.float32)
    with decode_policy("rows"):
        out = host(c.decode(dev(Q), dev(kl, torch.int32)))
    assert np.abs(out - O.decode(Q, K, V, kl)).max() <= TOL[cache_dtype]
