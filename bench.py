#!/usr/bin/env python
"""Benchmark of the cross-attention hot path on batched Whisper-Base windows.

One step = one window of the workload: populate the K/V projection cache of
B = 16 encoder memories (E_b [1500, 512], 6 layers, 8 heads x 64, ragged
key_len ~ U{500..1500}), then 128 decode steps, each one query row per (slot,
layer, head) over the cache. Throughput is decode tokens/s over the whole
window (a token = one query row per slot through all 6 layers' cross-attention),
populate included. Inputs are seeded synthetic tensors resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cxa|reference]

--impl reference times the fp64 CPU oracle on the host cores (a bounded sample
of the same workload per step). Under torchrun each rank runs its own replica of
the workload on its own GPU (weak scaling, no data-path collective); rank 0
prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "batched_base"
NOMINAL_HBM_GBS = 7900.0
TF32_OVER_BF16 = 0.5                 # dense TF32 / bf16 tensor rate (ncu: 4096 vs 8192 FLOP/clk/SM)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "decode_traffic.json")


# ---------------------------------------------------------------- host helpers
def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["cxa", "reference"], default="cxa")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    p.add_argument("--no-variants", action="store_true", help="skip the bf16-cache variant")
    p.add_argument("--profile", choices=["decode", "decode_bf16", "populate", "shared_bf16", "shared_bf16_16", "shared_f32",
                                          "align", "block", "selfattn", "decode_single", "decode_single_bf16"],
                   default=None,
                   help="run a few launches of one kernel on the workload's inputs (for ncu), print nothing else")
    p.add_argument("--sweep", action="store_true",
                   help="time decode and populate at every point of the decode bandwidth sweep "
                        "(T_enc x batch, d=512, 6 layers, 8x64 heads); one JSON line per point")
    p.add_argument("--shared", action="store_true",
                   help="time shared-cache decode (nq hypotheses per memory) on the batched Whisper-Base "
                        "workload for nq = 1, 2, 4, 5, 8 (and 12, 16 with a bf16 cache); one JSON line per "
                        "(nq, cache dtype)")
    p.add_argument("--small", action="store_true",
                   help="Whisper-Tiny / Whisper-Base single-memory decode, warm-L2 and cold, and populate")
    p.add_argument("--block", action="store_true",
                   help="time the per-layer cross-attention block (LayerNorm, Q projection, attention, out "
                        "projection + residual) for all 6 layers of a batched Whisper-Base decode step")
    p.add_argument("--selfattn", action="store_true",
                   help="time the self-attention KV-cache step (append + decode over positions 0..pos) over a "
                        "full 448-token sequence of the batched Whisper-Base decoder (16 slots, 6 layers, 8x64)")
    p.add_argument("--align", action="store_true",
                   help="time the alignment-head weights call on batched Whisper-Base (6 heads) and "
                        "Whisper-large dims (16 heads)")
    p.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--oracle-subset", choices=["large", "sweep"], default=None, help=argparse.SUPPRESS)
    p.add_argument("--oracle-small", choices=["tiny", "base"], default=None, help=argparse.SUPPRESS)
    p.add_argument("--save", default=None, help=argparse.SUPPRESS)
    p.add_argument("--budget-s", type=float, default=12.0, help=argparse.SUPPRESS)
    p.add_argument("--max-slots", type=int, default=16, help=argparse.SUPPRESS)
    p.add_argument("--procs", type=int, default=1, help=argparse.SUPPRESS)
    a = p.parse_args(argv)
    if a.warmup < 3 and not (a.oracle_sample or a.oracle_subset or a.oracle_small):
        p.error("--warmup must be >= 3")
    return a


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_slots(rank: int, B: int):
    """Seed indices of the encoder memories a rank owns: each rank runs its own
    B windows (weak scaling), distinct across ranks."""
    return list(range(rank * B, rank * B + B))


def max_over_ranks(dist, values, device):
    """Element-wise max of per-rank timings (the slowest rank sets the job time)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        pk["source"] = "measured"
        return pk
    except (OSError, ValueError):
        pk = dict(FALLBACK_PEAKS)
        pk["source"] = "fallback"
        return pk


def decode_bytes(L, H, dh, cache_esz, key_len, B):
    """Algorithmic bytes of one decode launch: K and V rows of the valid keys,
    the query rows read and the output rows written."""
    return 2 * L * H * dh * cache_esz * int(sum(int(k) for k in key_len)) + 2 * B * L * H * dh * 4


def populate_flops(L, d, B, T):
    """K and V projections of every row of every memory: 2 * (2*L*d) * d * B*T."""
    return 4 * L * d * d * B * T


DECODE_SOURCES = ("decode.cu", "chunk_stream.cuh", "ptx.cuh", "internal.h")


def source_sha(paths):
    """First 16 hex digits of the SHA-256 over the given files, concatenated in order."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """Per-launch DRAM bytes of the decode kernel from the committed ncu figure
    (profiles/decode_traffic.json), valid only while the kernel's sources hash to
    the value recorded with it."""
    try:
        with open(TRAFFIC_JSON) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    srcs = [os.path.join(ROOT, "encoder_decoder_speech_gb300", "csrc", f) for f in rec.get("sources", DECODE_SOURCES)]
    try:
        if source_sha(srcs) != rec.get("source_sha256_16"):
            return None
    except OSError:
        return None
    return float(rec["traffic_bytes_per_launch"])


def provenance():
    """What produced the line: the git commit (when the tree is a checkout), a hash
    of the product sources (always), and the driver, CUDA and torch versions."""
    def run(cmd):
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=20, cwd=ROOT)
            return r.stdout.strip() if r.returncode == 0 else None
        except (OSError, subprocess.SubprocessError):
            return None
    import glob
    files = sorted(glob.glob(os.path.join(ROOT, "encoder_decoder_speech_gb300", "csrc", "*")) +
                   glob.glob(os.path.join(ROOT, "include", "*.h")) +
                   [os.path.join(ROOT, "bench.py"), os.path.join(ROOT, "encoder_decoder_speech_gb300", "cxa.py")])
    nvcc = run(["nvcc", "--version"]) or run(["/usr/local/cuda/bin/nvcc", "--version"])
    out = {"git_sha": run(["git", "rev-parse", "HEAD"]), "source_sha256_16": source_sha(files),
           "driver": run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader", "-i", "0"]),
           "nvcc": next((x.strip() for x in nvcc.splitlines() if "release" in x), None) if nvcc else None}
    try:
        import torch
        out["torch"] = torch.__version__
        out["torch_cuda"] = torch.version.cuda
    except ImportError:
        pass
    return out


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm = []
        for r in rows:
            try:
                sm.append(float(r[1]))
            except ValueError:
                pass
            for i, n in enumerate(names):
                if r[5 + i].lower() == "active":
                    reasons.add(n)
        sm.sort()
        try:
            smax = float(rows[-1][2])
        except ValueError:
            smax = None
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- oracle legs
def oracle_sample(budget_s: float, max_slots: int, warmup_slots: int = 0, first_slot: int = 0,
                  save_path: str | None = None):
    """Time the fp64 oracle on whole windows of the workload (one memory: its
    populate, then its 128 decode steps), one memory after another, until
    max_slots windows are timed or the time budget is spent. warmup_slots
    windows run first, untimed. With save_path, the first timed window's 128
    decode outputs are saved there (for the informational PSNR of the GPU's
    outputs against them). Returns tokens, seconds, slots."""
    import numpy as np
    from encoder_decoder_speech_gb300 import workloads as W
    from oracle import cross_attention as O
    w = W.WORKLOADS[WORKLOAD]
    WK, WV, bV = W.make_weights(w)
    kl_all = W.make_key_len(w)
    Qs = [W.make_Q(w, s) for s in range(w.steps)]

    def window(b, keep=None):
        E = W.make_E(w, b, kl_all)[None]
        t0 = time.perf_counter()
        Kc, Vc = O.populate(E, WK, WV, bV, w.H)
        for s in range(w.steps):
            o = O.decode(Qs[s][b:b + 1], Kc, Vc, kl_all[b:b + 1])
            if keep is not None:
                keep.append(o[0])
        return time.perf_counter() - t0

    for i in range(warmup_slots):
        window((first_slot + i) % w.B)
    tokens, slots, spent = 0, 0, 0.0
    for i in range(max_slots):
        keep = [] if (save_path and i == 0) else None
        spent += window((first_slot + i) % w.B, keep)
        if keep is not None:
            np.save(save_path, np.stack(keep))
        tokens += w.steps
        slots += 1
        if spent >= budget_s:
            break
    return {"tokens": tokens, "seconds": spent, "slots": slots, "saved_slot": first_slot % w.B if save_path else None}


def oracle_subset(which: str, budget_s: float):
    """The oracle on a labelled subset of a workload too large to run whole: random
    (slot, layer, head) units, each its own K/V projection (the head's column block
    of the GEMM) plus every decode step of its query row over its keys. Reports the
    time per unit and the whole window projected from it (units x time per unit)."""
    import numpy as np
    from encoder_decoder_speech_gb300 import workloads as W
    from oracle import cross_attention as O
    if which == "large":
        w = W.WORKLOADS["large"]
        steps = w.steps
    else:
        w = W.sweep_workload(32768, 64)
        steps = w.steps
    WK, WV, bV = W.make_weights(w)
    kl = W.make_key_len(w)
    rng = np.random.default_rng(5)
    units_total = w.B * w.L * w.H
    spent, units = 0.0, 0
    while spent < budget_s and units < 64:
        b, l, h = int(rng.integers(w.B)), int(rng.integers(w.L)), int(rng.integers(w.H))
        E = W.make_E(w, b, kl)
        q = np.stack([W.make_Q(w, s)[b, l, h] for s in range(steps)])
        t0 = time.perf_counter()
        K, V = O.populate_head(E, WK[l], WV[l], bV[l], h)
        for s in range(steps):
            O.attend_row(q[s], K, V, int(kl[b]), w.scale)
        spent += time.perf_counter() - t0
        units += 1
    per_unit = spent / units
    window_s = per_unit * units_total
    return {"workload": ("whisper-large dims: 8 x [1500,1280], 32 layers x 20 heads, 256 decode steps"
                         if which == "large" else "sweep T_enc 32768 x B 64, d 512, 6 layers x 8 heads, 100 steps"),
            "kind": "oracle", "subset": f"{units} of {units_total} (slot, layer, head) units, chosen at random",
            "seconds_per_unit": per_unit, "projected_window_s": window_s,
            "projected_tokens_per_s": w.B * steps / window_s, "cores": 1}


def _oracle_worker(args):
    budget_s, max_slots, first_slot = args
    return oracle_sample(budget_s, max_slots, 1, first_slot)


def oracle_sample_procs(budget_s: float, max_slots: int, procs: int):
    """The same windows on procs worker processes at once (started with spawn, each
    single-threaded): windows are independent, so this is the oracle as it stands
    on procs host cores. Returns tokens over the wall time of the timed windows."""
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(procs) as pool:
        pool.map(_oracle_worker, [(0.0, 0, i) for i in range(procs)])   # imports and first window untimed
        t0 = time.perf_counter()
        res = pool.map(_oracle_worker, [(budget_s, max_slots, i) for i in range(procs)])
        wall = time.perf_counter() - t0
    return {"tokens": sum(r["tokens"] for r in res), "seconds": wall, "slots": sum(r["slots"] for r in res),
            "procs": procs}


def cpu_model() -> str:
    """The host CPU's model name as the OS reports it (best effort)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_small_window(name: str):
    """The oracle on one whole window of a single-memory workload (Whisper-Tiny dims:
    populate + 1 step; Whisper-Base dims: populate + 64 steps), single-threaded."""
    from encoder_decoder_speech_gb300 import workloads as W
    from oracle import cross_attention as O
    w = W.WORKLOADS[name]
    E = W.make_E_all(w)
    WK, WV, bV = W.make_weights(w)
    kl = W.make_key_len(w)
    Qs = [W.make_Q(w, s) for s in range(w.steps)]
    t0 = time.perf_counter()
    Kc, Vc = O.populate(E, WK, WV, bV, w.H)
    t1 = time.perf_counter()
    for s in range(w.steps):
        O.decode(Qs[s], Kc, Vc, kl)
    t2 = time.perf_counter()
    return {"kind": "oracle", "cores": 1, "workload": name, "window_s": t2 - t0, "populate_s": t1 - t0,
            "decode_s_per_step": (t2 - t1) / w.steps, "tokens_per_s": w.B * w.steps / (t2 - t0),
            "sample": f"one whole window: fp64 populate + {w.steps} decode step(s), single thread"}


def _oracle_env():
    return dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
                RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")


def run_oracle_subprocess(budget_s: float, max_slots: int, warmup_slots: int = 0, procs: int = 1,
                          save_path: str | None = None):
    """The oracle timed in a fresh process (BLAS pinned to one thread per process),
    single-threaded or on procs worker processes."""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--budget-s", str(budget_s),
           "--max-slots", str(max_slots), "--warmup", str(warmup_slots), "--procs", str(procs)]
    if save_path:
        cmd += ["--save", save_path]
    r = subprocess.run(cmd, capture_output=True, text=True, env=_oracle_env(), timeout=3600)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_oracle_subset_subprocess(which: str, budget_s: float):
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-subset", which, "--budget-s",
                        str(budget_s), "--warmup", "0"], capture_output=True, text=True, env=_oracle_env(),
                       timeout=3600)
    if r.returncode != 0:
        raise RuntimeError("oracle subset failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_obj(res):
    procs = res.get("procs", 1)
    how = "single thread" if procs == 1 else f"{procs} single-threaded processes at once, wall time"
    return {"value": res["tokens"] / res["seconds"], "unit": "tokens/s", "cores": procs, "kind": "oracle",
            "sample": f"{res['slots']} whole window(s) of the workload (one memory each: fp64 populate + "
                      f"128 decode steps), {res['tokens']} tokens in {res['seconds']:.1f} s, {how}",
            "cpu_model": cpu_model(), "nproc": os.cpu_count()}


def run_reference(args):
    """The oracle as the reference arm: each step is one whole window of one
    memory (populate + 128 decode steps), W untimed then K timed."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from encoder_decoder_speech_gb300 import workloads as W
    w = W.WORKLOADS[WORKLOAD]
    res = run_oracle_subprocess(budget_s=float("inf"), max_slots=args.steps, warmup_slots=args.warmup)
    value = res["tokens"] / res["seconds"]
    line = {
        "impl": "reference",
        "metric": "cross-attn decode tokens/s (batched Whisper-Base window: populate + 128 decode steps)",
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * res["seconds"] / max(res["slots"], 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy, Whisper-Base shapes)",
        "config": dict(workload_config(w, "f64 (oracle)"), populate_inputs="fp32 inputs, fp64 arithmetic (oracle)",
                       l2="host memory (the oracle runs on the CPU)"),
        "cpu_baseline": cpu_baseline_obj(res),
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(w, cache_dtype):
    return {"workload": "batched-whisper-base", "B": w.B, "T_enc": w.T, "d": w.d, "L": w.L, "H": w.H, "dh": w.dh,
            "decode_steps_per_window": w.steps, "key_len": "U{500..1500} per memory, padded rows zeroed",
            "cache_dtype": cache_dtype, "populate_inputs": "fp32 (TF32 tensor-core operands)",
            "l2": "inputs larger than L2: each decode step reads the valid K/V rows of a 590 MB fp32 cache "
                  "(394 MB), each populate writes 590 MB; no flush needed"}


# ---------------------------------------------------------------- GPU arm
def measure(torch, cxa, W, w, dev_inputs, cache_dtype, K, Wu, rank, world, dist, timed_clocks: bool):
    """Times K windows; returns a dict of timings (max over ranks)."""
    E, WK, WV, bV, kl, Qs, key_len_host = dev_inputs
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, cache_dtype)
    out = torch.empty((w.B, w.L, w.H, w.dh), dtype=torch.float32, device="cuda")
    h = cache.handle
    # the layer weights are the model's: packed once, when they are loaded, and
    # every window's populate is then one GEMM over the packed copy
    packed = cache.pack_weights(WK, WV, stream=sptr)

    def pack():
        cxa.check(cxa.cxa_pack_weights(WK, WV, w.d, w.L, cxa.CXA_F32, packed, packed.numel(), sptr),
                  "cxa_pack_weights")

    def populate():
        cxa.check(cxa.cxa_populate_packed(h, 0, w.B, E, packed, packed.numel(), bV, w.T, w.d, w.L, w.H,
                                          cxa.CXA_F32, sptr), "cxa_populate_packed")

    def decode(s):
        cxa.check(cxa.cxa_decode(h, Qs[s], kl, out, 0.0, cache.decode_ws, cache.decode_ws_bytes, sptr), "cxa_decode")

    for _ in range(Wu):
        populate()
        for s in range(w.steps):
            decode(s)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(torch.cuda.current_device()) if timed_clocks else None
    if clk:
        clk.start()
    launches0 = cxa.cxa_launch_count()
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(K):
        ev[k][0].record(stream)
        populate()
        ev[k][1].record(stream)
        for s in range(w.steps):
            decode(s)
        ev[k][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = cxa.cxa_launch_count() - launches0
    clocks = clk.stop() if clk else None
    if dist is not None:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    pop_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    if dist is not None:
        total_ms, pop_ms, dec_ms = max_over_ranks(dist, [total_ms, pop_ms, dec_ms], "cuda")
    assert cxa.cxa_device_status(1) == cxa.CXA_OK, "a kernel reported a bounded-wait timeout"
    # the one-time weight packing, timed on its own (10 calls)
    pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pa.record(stream)
    for _ in range(10):
        pack()
    pb.record(stream)
    torch.cuda.synchronize()
    pack_ms = pa.elapsed_time(pb) / 10
    res = {"total_ms": total_ms, "populate_ms": pop_ms, "decode_window_ms": dec_ms, "pack_weights_ms": pack_ms,
           "decode_launch_us": 1000.0 * dec_ms / w.steps, "launches": launches, "clocks": clocks}
    # spread over the K windows (this rank's events): window, populate and decode-loop times
    import numpy as np

    def pct(xs):
        a = np.asarray(xs, dtype=np.float64)
        return {"p10": round(float(np.percentile(a, 10)), 4), "median": round(float(np.median(a)), 4),
                "p90": round(float(np.percentile(a, 90)), 4), "n": int(a.size)}

    res["spread_ms"] = {"window": pct([e[0].elapsed_time(e[2]) for e in ev]),
                        "populate": pct([e[0].elapsed_time(e[1]) for e in ev]),
                        "decode_128_steps": pct([e[1].elapsed_time(e[2]) for e in ev])}
    cache.close()
    return res


def measure_e2e(torch, cxa, w, host_inputs, dev_static, K, Wu, dist):
    """Same windows through the public API with inputs in pinned host memory. Every
    window copies in its E, key_len and its 128 steps' Q, and copies out its 128
    steps' outputs. A copy stream double-buffers: window k+1's inputs move in and
    window k-1's outputs move out while window k computes (CUDA events order the
    two streams)."""
    E_h, kl_h, Q_h = host_inputs
    WK, WV, bV = dev_static
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    E_pin = torch.from_numpy(E_h).pin_memory()
    kl_pin = torch.from_numpy(kl_h).pin_memory()
    Q_pin = torch.from_numpy(Q_h).pin_memory()
    out_pin = torch.empty((w.steps, w.B, w.L, w.H, w.dh), dtype=torch.float32).pin_memory()
    E_d = [torch.empty(E_pin.shape, dtype=torch.float32, device="cuda") for _ in range(2)]
    kl_d = [torch.empty(kl_pin.shape, dtype=torch.int32, device="cuda") for _ in range(2)]
    Q_d = [torch.empty(Q_pin.shape, dtype=torch.float32, device="cuda") for _ in range(2)]
    out_d = [torch.empty(out_pin.shape, dtype=torch.float32, device="cuda") for _ in range(2)]
    inputs_ready = [torch.cuda.Event() for _ in range(2)]
    outputs_ready = [torch.cuda.Event() for _ in range(2)]
    buffers_free = [torch.cuda.Event() for _ in range(2)]
    cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, "f32")
    h = cache.handle
    sptr = comp.cuda_stream
    packed = cache.pack_weights(WK, WV, stream=sptr)      # once, with the model weights

    def stage_in(k):
        i = k % 2
        with torch.cuda.stream(copy):
            copy.wait_event(buffers_free[i])
            E_d[i].copy_(E_pin, non_blocking=True)
            kl_d[i].copy_(kl_pin, non_blocking=True)
            Q_d[i].copy_(Q_pin, non_blocking=True)
            inputs_ready[i].record(copy)

    def compute(k):
        i = k % 2
        comp.wait_event(inputs_ready[i])
        cxa.check(cxa.cxa_populate_packed(h, 0, w.B, E_d[i], packed, packed.numel(), bV, w.T, w.d, w.L, w.H,
                                          cxa.CXA_F32, sptr), "cxa_populate_packed")
        for s in range(w.steps):
            cxa.check(cxa.cxa_decode(h, Q_d[i][s], kl_d[i], out_d[i][s], 0.0, cache.decode_ws, cache.decode_ws_bytes,
                                     sptr), "cxa_decode")
        outputs_ready[i].record(comp)

    def stage_out(k):
        i = k % 2
        with torch.cuda.stream(copy):
            copy.wait_event(outputs_ready[i])
            out_pin.copy_(out_d[i], non_blocking=True)
            buffers_free[i].record(copy)

    def run(n):
        for i in range(2):
            buffers_free[i].record(copy)
        stage_in(0)
        for k in range(n):
            if k + 1 < n:
                stage_in(k + 1)
            compute(k)
            stage_out(k)
        comp.wait_stream(copy)

    run(Wu)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    # three timed runs of K windows; the median is reported (a host that is briefly
    # busy slows the copies of one run, not the others)
    reps = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        run(K)
        b.record(comp)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        if dist is not None:
            ms = max_over_ranks(dist, [ms], "cuda")[0]
        reps.append(ms)
    h2d = E_pin.numel() * 4 + kl_pin.numel() * 4 + Q_pin.numel() * 4
    d2h = out_pin.numel() * 4
    cache.close()
    return sorted(reps)[1], h2d, d2h, reps


def device_inputs(torch, W, w, rank):
    """Seeded inputs of the workload for this rank, uploaded to the current GPU."""
    import numpy as np
    kl = W.make_key_len(w)
    E = np.stack([W.make_E(W.replace(w, ragged=False), s) for s in rank_slots(rank, w.B)])
    for i in range(w.B):                      # pad rows of each memory are zero
        E[i, int(kl[i]):] = 0.0
    WK, WV, bV = W.make_weights(w)
    Q = np.stack([W.make_Q(w, s) for s in range(w.steps)])

    def d(x, dt=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dt)

    return (d(E), d(WK), d(WV), d(bV), d(kl, torch.int32), d(Q), kl), (E, kl.astype(np.int32), Q)


def measure_populate_large(torch, cxa, W, Wu, reps=10):
    """Whisper-large dims (8 memories [1500, 1280], 32 layers, 20 heads): the
    encoder memory arrives in fp32 and is converted to bf16 on the device
    (cxa_convert_bf16, timed apart); the weights are converted and packed once;
    the populate GEMM runs on bf16 tensor cores into a bf16 cache (the bf16
    tensor-core roofline is quoted on it)."""
    import numpy as np
    w = W.WORKLOADS["large"]
    wf = W.replace(w, in_dtype="f32")                      # the same draws, not rounded on the host
    E32 = torch.from_numpy(W.make_E_all(wf)).to("cuda")
    WK32, WV32, bV = W.make_weights(wf)
    WK32, WV32 = torch.from_numpy(WK32).to("cuda"), torch.from_numpy(WV32).to("cuda")
    bV = torch.from_numpy(np.ascontiguousarray(bV)).to("cuda")
    cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, "bf16")
    E = cxa.to_bf16(E32)
    packed = cache.pack_weights(cxa.to_bf16(WK32), cxa.to_bf16(WV32))
    del WK32, WV32
    for _ in range(Wu):
        cxa.to_bf16(E32, out=E)
        cache.populate_packed(E, packed, bV)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c = torch.cuda.Event(enable_timing=True)
    # the conversion alone, back to back (timed from an idle GPU, one call would also
    # count the host's launch of it)
    a.record()
    for _ in range(reps):
        cxa.to_bf16(E32, out=E)
    b.record()
    torch.cuda.synchronize()
    conv_ms = a.elapsed_time(b) / reps
    # each populate right behind its conversion (its launch queues while that runs)
    pop_ms = 0.0
    for _ in range(reps):
        cxa.to_bf16(E32, out=E)
        b.record()
        cache.populate_packed(E, packed, bV)
        c.record()
        torch.cuda.synchronize()
        pop_ms += b.elapsed_time(c) / reps
    ms = pop_ms
    # the workload's 256 decode steps on the same cache, each a fresh query set:
    # 8 x 32 x 20 query rows over 1500 keys each (1.97 GB of K/V per step)
    kl_h = W.make_key_len(w)
    kl = torch.from_numpy(kl_h).to("cuda")
    steps = w.steps
    Qs = torch.from_numpy(np.stack([W.make_Q(w, s) for s in range(steps)])).to("cuda")
    out = torch.empty_like(Qs[0])
    for s in range(max(Wu, 3)):
        cache.decode(Qs[s], kl, out=out)
    torch.cuda.synchronize()
    a.record()
    for s in range(steps):
        cache.decode(Qs[s], kl, out=out)
    b.record()
    torch.cuda.synchronize()
    dec_us = a.elapsed_time(b) * 1000.0 / steps
    cache.close()
    return {"ms": ms, "flops_per_call": populate_flops(w.L, w.d, w.B, w.T), "decode_us": dec_us,
            "decode_bytes": decode_bytes(w.L, w.H, w.dh, 2, kl_h, w.B), "B": w.B, "convert_ms": conv_ms,
            "convert_bytes": E32.numel() * 6, "steps": steps, "T": w.T, "d": w.d, "L": w.L}


def run_sweep(args):
    """Decode bandwidth sweep: every (T_enc, batch) point, fp32 and bf16 caches,
    `--steps` timed decode steps after `--warmup` (CUDA events around the step
    loop, programmatic launch overlap included) and one timed populate."""
    import numpy as np
    import torch
    from encoder_decoder_speech_gb300 import _build, cxa
    from encoder_decoder_speech_gb300 import workloads as W
    _build.build_library()
    cxa.load()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    for T in W.SWEEP_T:
        for B in W.SWEEP_B:
            w = W.sweep_workload(T, B)
            WK, WV, bV = (torch.from_numpy(np.ascontiguousarray(x)).to("cuda") for x in W.make_weights(w))
            kl_h = W.make_key_len(w)
            kl = torch.from_numpy(kl_h).to("cuda")
            E = torch.empty((B, T, w.d), dtype=torch.float32, device="cuda")
            for b in range(B):
                E[b].copy_(torch.from_numpy(W.make_E(w, b, kl_h)))
            Q = torch.from_numpy(W.make_Q(w, 0)).to("cuda")
            line = {"sweep_point": {"T_enc": T, "B": B, "d": w.d, "L": w.L, "H": w.H}}
            for cd, esz in (("f32", 4), ("bf16", 2)):
                cache = cxa.CrossAttentionCache(B, T, w.L, w.H, 64, cd)
                out = torch.empty_like(Q)
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                packed = cache.pack_weights(WK, WV)
                cache.populate_packed(E, packed, bV)
                torch.cuda.synchronize()
                a.record()
                cache.populate_packed(E, packed, bV)
                b_.record()
                torch.cuda.synchronize()
                pop_ms = a.elapsed_time(b_)
                for _ in range(args.warmup):
                    cache.decode(Q, kl, out=out)
                torch.cuda.synchronize()
                a.record()
                for _ in range(args.steps):
                    cache.decode(Q, kl, out=out)
                b_.record()
                torch.cuda.synchronize()
                us = a.elapsed_time(b_) * 1000.0 / args.steps
                gbs = decode_bytes(w.L, w.H, w.dh, esz, kl_h, B) / (us * 1e-6) / 1e9
                line[cd] = {"decode_us": round(us, 2), "decode_GBps": round(gbs, 1),
                            "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 3),
                            "tokens_per_s": round(B / (us * 1e-6), 1), "populate_ms": round(pop_ms, 4),
                            "populate_TFLOPs": round(populate_flops(w.L, w.d, B, T) / (pop_ms * 1e-3) / 1e12, 1)}
                cache.close()
                del cache
                torch.cuda.empty_cache()
            assert cxa.cxa_device_status(1) == cxa.CXA_OK
            print(json.dumps(line), flush=True)
            del E
            torch.cuda.empty_cache()
    return 0


def run_shared(args):
    """Shared-cache decode on batched Whisper-Base: nq hypothesis rows per memory
    read the memory's K/V once. A token here is one query row of one hypothesis
    through all layers; bytes = valid K/V rows + nq x (Q + out) rows."""
    import numpy as np
    import torch
    from encoder_decoder_speech_gb300 import _build, cxa
    from encoder_decoder_speech_gb300 import workloads as W
    _build.build_library()
    cxa.load()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    w = W.WORKLOADS[WORKLOAD]
    (E, WK, WV, bV, kl, _, kl_h), _ = device_inputs(torch, W, w, 0)
    for cd, esz in (("f32", 4), ("bf16", 2)):
        cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, cd)
        cache.populate(E, WK, WV, bV)
        for nq in (1, 2, 4, 5, 8) + ((12, 16) if cd == "bf16" else ()):
            Q = torch.from_numpy(np.random.default_rng(nq).standard_normal(
                (w.B, nq, w.L, w.H, w.dh)).astype(np.float32)).to("cuda")
            out = torch.empty_like(Q)
            for _ in range(args.warmup):
                cache.decode_shared(Q, kl, out=out)
            torch.cuda.synchronize()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(args.steps):
                cache.decode_shared(Q, kl, out=out)
            b_.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b_) * 1000.0 / args.steps
            byts = decode_bytes(w.L, w.H, w.dh, esz, kl_h, w.B) + (nq - 1) * 2 * w.B * w.L * w.H * w.dh * 4
            print(json.dumps({"shared_decode": {"workload": "batched-whisper-base", "nq": nq, "cache_dtype": cd},
                              "us_per_step": round(us, 2), "tokens_per_s": round(w.B * nq / (us * 1e-6), 1),
                              "GBps": round(byts / (us * 1e-6) / 1e9, 1),
                              "frac_of_measured_hbm": round(byts / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3)}),
                  flush=True)
        cache.close()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK
    return 0


def run_small(args):
    """The single-memory configurations (Whisper-Tiny dims, Whisper-Base dims): their
    fp32 caches (18-37 MB of valid K/V) fit in the 129 MB L2, so each decode is timed
    warm (steps back to back, the cache stays in L2; launched from Python one by one,
    and replayed from a CUDA graph) and cold (each step after a 512 MB read that
    evicts the cache; graph of read + step pairs minus a graph of the reads alone),
    for the automatic kernel choice and the persistent stream kernel; the populate
    from weights packed once is timed back to back (20 calls) and cold (mean of 20,
    CUDA events, launch latency included)."""
    import numpy as np
    # the oracle on one window of each workload, in its own process, before any GPU work
    oracle = {}
    if not args.no_cpu_baseline:
        for name in ("tiny", "base"):
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-small", name, "--warmup", "0"],
                               capture_output=True, text=True, env=_oracle_env(), timeout=1800)
            if r.returncode == 0:
                oracle[name] = json.loads(r.stdout.strip().splitlines()[-1])
    import torch
    from encoder_decoder_speech_gb300 import _build, cxa
    from encoder_decoder_speech_gb300 import workloads as W
    _build.build_library()
    cxa.load()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for name in ("tiny", "base"):
        w = W.WORKLOADS[name]
        (E, WK, WV, bV, kl, Qs, kl_h), _ = device_inputs(torch, W, w, 0)
        for cd, esz in (("f32", 4), ("bf16", 2)):
            cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, cd)
            out = torch.empty((w.B, w.L, w.H, w.dh), device="cuda")
            packed = cache.pack_weights(WK, WV)
            for _ in range(args.warmup):
                cache.populate_packed(E, packed, bV)
            torch.cuda.synchronize()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(20):
                cache.populate_packed(E, packed, bV)
            b_.record()
            torch.cuda.synchronize()
            pop_ms = a.elapsed_time(b_) / 20
            pop_cold = []
            for s in range(20):
                flush.view(torch.int64).sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                cache.populate_packed(E, packed, bV)
                e1.record()
                torch.cuda.synchronize()
                pop_cold.append(e0.elapsed_time(e1))
            n = args.steps
            byts = decode_bytes(w.L, w.H, w.dh, esz, kl_h, w.B)
            res = {}
            for shape, pol in (("auto", cxa.CXA_DECODE_AUTO), ("stream", cxa.CXA_DECODE_STREAM)):
                cxa.check(cxa.cxa_set_decode_policy(pol), "cxa_set_decode_policy")
                for s in range(args.warmup):
                    cache.decode(Qs[s % Qs.shape[0]], kl, out=out)
                torch.cuda.synchronize()
                a.record()
                for s in range(n):
                    cache.decode(Qs[s % Qs.shape[0]], kl, out=out)
                b_.record()
                torch.cuda.synchronize()
                warm_us = a.elapsed_time(b_) * 1000.0 / n
                # the same steps replayed from a CUDA graph (64 steps per graph)
                g = torch.cuda.CUDAGraph()
                gs = torch.cuda.Stream()
                gs.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(gs):
                    with torch.cuda.graph(g, stream=gs):
                        for s in range(64):
                            cache.decode(Qs[s % Qs.shape[0]], kl, out=out, stream=gs)
                torch.cuda.synchronize()
                g.replay()
                torch.cuda.synchronize()
                a.record()
                reps = max(1, n // 64)
                for _ in range(reps):
                    g.replay()
                b_.record()
                torch.cuda.synchronize()
                graph_us = a.elapsed_time(b_) * 1000.0 / (64 * reps)
                del g
                # cold: each step right after a 512 MB read that leaves only clean lines of
                # other data in L2; 32 (read, step) pairs in a graph minus 32 reads alone
                # (no host launch latency in either, and no timer quantisation)
                def pairs(with_step):
                    gg = torch.cuda.CUDAGraph()
                    with torch.cuda.stream(gs):
                        with torch.cuda.graph(gg, stream=gs):
                            for s in range(32):
                                flush.view(torch.int64).sum()
                                if with_step:
                                    cache.decode(Qs[s % Qs.shape[0]], kl, out=out, stream=gs)
                    torch.cuda.synchronize()
                    gg.replay()
                    torch.cuda.synchronize()
                    a.record()
                    for _ in range(5):
                        gg.replay()
                    b_.record()
                    torch.cuda.synchronize()
                    return a.elapsed_time(b_) * 1000.0 / (5 * 32)
                cold_us = pairs(True) - pairs(False)
                res[shape] = {"decode_us_warm_l2": round(warm_us, 2), "decode_us_graph_warm_l2": round(graph_us, 2),
                              "decode_us_cold": round(cold_us, 2),
                              "decode_GBps_cold": round(byts / (cold_us * 1e-6) / 1e9, 1),
                              "frac_of_measured_hbm_cold": round(byts / (cold_us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3)}
            cxa.check(cxa.cxa_set_decode_policy(cxa.CXA_DECODE_AUTO), "cxa_set_decode_policy")
            print(json.dumps({"small_config": {"workload": name, "T_enc": w.T, "d": w.d, "L": w.L, "H": w.H,
                                               "cache_dtype": cd},
                              **res["auto"], "stream_kernel": res["stream"],
                              "populate_ms": round(pop_ms, 4),
                              "populate_TFLOPs": round(populate_flops(w.L, w.d, w.B, w.T) / (pop_ms * 1e-3) / 1e12, 1),
                              "populate_ms_cold": round(float(np.mean(pop_cold)), 4),
                              "cpu_baseline": oracle.get(name)}),
                  flush=True)
            cache.close()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK
    return 0


def run_block(args):
    """One decoder step of batched Whisper-Base through the per-layer entry point:
    for l = 0..5, x = x + CrossAttn_l(LayerNorm(x)) (cxa_cross_block), fp32 weights."""
    import numpy as np
    import torch
    from encoder_decoder_speech_gb300 import _build, cxa
    from encoder_decoder_speech_gb300 import workloads as W
    _build.build_library()
    cxa.load()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    w = W.WORKLOADS[WORKLOAD]
    (E, WK, WV, bV, kl, _, kl_h), _ = device_inputs(torch, W, w, 0)
    rng = np.random.default_rng(5)

    def t(shape, std):
        return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to("cuda")

    prm = [dict(WQ=t((w.d, w.d), w.d ** -0.5), WO=t((w.d, w.d), w.d ** -0.5), g=1 + t((w.d,), 0.1),
                b=t((w.d,), 0.1), bQ=t((w.d,), 0.02), bO=t((w.d,), 0.02)) for _ in range(w.L)]
    for cd, esz in (("f32", 4), ("bf16", 2)):
        cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, cd)
        cache.populate(E, WK, WV, bV)
        x = t((w.B, w.d), 1.0)

        def step():
            for l in range(w.L):
                p = prm[l]
                cache.cross_block(l, x, p["WQ"], p["WO"], kl, ln_gamma=p["g"], ln_beta=p["b"], bQ=p["bQ"], bO=p["bO"])

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        byts = decode_bytes(w.L, w.H, w.dh, esz, kl_h, w.B) + w.L * 2 * w.d * w.d * 4 + w.L * 3 * w.B * w.d * 4
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # launched one call at a time from Python, then replayed as one captured CUDA graph per step
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        n0 = cxa.cxa_launch_count()
        step()
        torch.cuda.synchronize()
        kernels_per_step = cxa.cxa_launch_count() - n0
        for mode in ("eager", "graph"):
            run = step if mode == "eager" else graph.replay
            for _ in range(args.warmup):
                run()
            torch.cuda.synchronize()
            a.record()
            for _ in range(args.steps):
                run()
            b_.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b_) * 1000.0 / args.steps
            print(json.dumps({"cross_block_step": {"workload": "batched-whisper-base", "layers": w.L,
                                                   "cache_dtype": cd, "launch": mode},
                              "us_per_step": round(us, 2), "tokens_per_s": round(w.B / (us * 1e-6), 1),
                              "GBps": round(byts / (us * 1e-6) / 1e9, 1),
                              "frac_of_measured_hbm": round(byts / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3),
                              "kernels_per_step": kernels_per_step}), flush=True)
        del graph
        cache.close()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK
    return 0


def run_selfattn(args):
    """Self-attention KV cache (max_seq_len 448): one token step = append the new
    K/V row at position pos in every (slot, layer, head), then decode positions
    0..pos. A whole 448-step sequence is timed (CUDA events around all steps),
    launched call by call and as one CUDA graph, and reported per step; bytes = K/V
    rows read + new rows written + Q and out."""
    import numpy as np
    import torch
    from encoder_decoder_speech_gb300 import _build, cxa
    from encoder_decoder_speech_gb300 import workloads as W
    _build.build_library()
    cxa.load()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    B, L, H, T = 16, 6, 8, 448
    rng = np.random.default_rng(11)
    Qs = torch.from_numpy(rng.standard_normal((T, B, L, H, 64)).astype(np.float32)).to("cuda")
    Ks = torch.from_numpy(rng.standard_normal((T, B, L, H, 64)).astype(np.float32)).to("cuda")
    Vs = torch.from_numpy(rng.standard_normal((T, B, L, H, 64)).astype(np.float32)).to("cuda")
    pos = [torch.full((B,), s, dtype=torch.int32, device="cuda") for s in range(T)]
    # per-step views made once, so that the eager loop times the library calls
    Qs, Ks, Vs = list(Qs.unbind(0)), list(Ks.unbind(0)), list(Vs.unbind(0))
    for cd, esz in (("f32", 4), ("bf16", 2)):
        cache = cxa.CrossAttentionCache(B, T, L, H, 64, cd)
        out = torch.empty((B, L, H, 64), device="cuda")

        def sequence():
            for s in range(T):
                cache.self_attention_step(pos[s], Qs[s], Ks[s], Vs[s], out=out)

        for s in range(min(args.warmup, T)):
            cache.self_attention_step(pos[s], Qs[s], Ks[s], Vs[s], out=out)
        torch.cuda.synchronize()
        n0 = cxa.cxa_launch_count()
        sequence()
        torch.cuda.synchronize()
        kernels_per_step = (cxa.cxa_launch_count() - n0) / T
        # the whole sequence launched one C-ABI call per step from Python, then
        # replayed as one captured CUDA graph (how a decoder loop would run it)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            sequence()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            sequence()
        torch.cuda.synchronize()
        rows = B * L * H
        byts = sum(2 * rows * (s + 1) * 64 * esz for s in range(T)) / T + rows * 64 * (2 * esz + 2 * 4 + 2 * 4)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for mode in ("eager", "graph"):
            run = sequence if mode == "eager" else graph.replay
            run()
            torch.cuda.synchronize()
            h0 = time.perf_counter()
            a.record()
            run()
            b_.record()
            h1 = time.perf_counter()
            torch.cuda.synchronize()
            us = a.elapsed_time(b_) * 1000.0 / T
            line = {"self_attention_step": {"B": B, "L": L, "H": H, "max_seq_len": T, "cache_dtype": cd,
                                            "launch": mode},
                    "us_per_step_mean": round(us, 2), "tokens_per_s": round(B / (us * 1e-6), 1),
                    "GBps_mean": round(byts / (us * 1e-6) / 1e9, 1),
                    "frac_of_measured_hbm": round(byts / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3),
                    "kernels_per_step": kernels_per_step}
            if mode == "eager":
                line["host_us_per_step"] = round((h1 - h0) * 1e6 / T, 2)
            print(json.dumps(line), flush=True)
        del graph
        # per position: a graph of 50 steps that all append and decode at one position
        per_pos = {}
        for ps in (0, 64, 256, T - 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                for s in range(3):
                    cache.self_attention_step(pos[ps], Qs[s], Ks[s], Vs[s], out=out, stream=side)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=side):
                for s in range(50):
                    cache.self_attention_step(pos[ps], Qs[s % 4], Ks[s % 4], Vs[s % 4], out=out, stream=side)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(4):
                g.replay()
            b_.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b_) * 1000.0 / 200
            kv = 2 * rows * (ps + 1) * 64 * esz
            per_pos[str(ps)] = {"us": round(us, 2), "kv_MB": round(kv / 1e6, 1), "GBps": round(kv / (us * 1e-6) / 1e9, 1)}
            del g
        print(json.dumps({"self_attention_step_per_position": {"cache_dtype": cd, "B": B, "L": L, "H": H,
                                                               "max_seq_len": T}, "positions": per_pos}), flush=True)
        cache.close()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK
    return 0


def run_align(args):
    """cxa_alignment_weights: softmax rows of selected (layer, head) pairs and their
    mean, per decode step. Bytes = K rows of the selected heads (valid keys) + the
    weights rows written (+ the mean)."""
    import numpy as np
    import torch
    from encoder_decoder_speech_gb300 import _build, cxa
    from encoder_decoder_speech_gb300 import workloads as W
    _build.build_library()
    cxa.load()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    for name, heads in (("batched_base", [(3, 1), (4, 2), (4, 6), (5, 0), (5, 3), (5, 7)]),
                        ("large", [(l, (7 * l) % 20) for l in range(16, 32)])):
        w = W.WORKLOADS[name]
        dt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
        cd = w.cache_dtypes[0]
        esz = 2 if cd == "bf16" else 4
        E = torch.randn(w.B, w.T, w.d, device="cuda").to(dt)
        WK = (torch.randn(w.L, w.d, w.d, device="cuda") / w.d ** 0.5).to(dt)
        bV = torch.zeros(w.L, w.d, device="cuda")
        kl_h = W.make_key_len(w)
        kl = torch.from_numpy(kl_h).to("cuda")
        cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, 64, cd)
        cache.populate(E, WK, WK, bV)
        Q = torch.randn(w.B, w.L, w.H, 64, device="cuda")
        wt = torch.empty((w.B, len(heads), w.T), device="cuda")
        mean = torch.empty((w.B, w.T), device="cuda")

        def call():
            cxa.check(cxa.cxa_alignment_weights(cache.handle, Q, kl, heads, wt, mean, 0.0), "align")

        per_graph = 50   # calls captured in one CUDA graph
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                call()
        torch.cuda.synchronize()
        n0 = cxa.cxa_launch_count()
        call()
        torch.cuda.synchronize()
        kernels_per_call = cxa.cxa_launch_count() - n0
        byts = len(heads) * 64 * esz * int(np.clip(kl_h, 0, w.T).sum()) + w.B * (len(heads) + 1) * w.T * 4 * 2
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for mode in ("eager", "graph"):
            reps = max(1, args.steps // per_graph) if mode == "graph" else args.steps
            run = call if mode == "eager" else graph.replay
            for _ in range(args.warmup):
                run()
            torch.cuda.synchronize()
            h0 = time.perf_counter()
            a.record()
            for _ in range(reps):
                run()
            b_.record()
            h1 = time.perf_counter()
            torch.cuda.synchronize()
            calls = reps * (per_graph if mode == "graph" else 1)
            us = a.elapsed_time(b_) * 1000.0 / calls
            line = {"alignment_weights": {"workload": name, "heads": len(heads), "cache_dtype": cd,
                                          "launch": mode},
                    "us_per_call": round(us, 2), "GBps": round(byts / (us * 1e-6) / 1e9, 1),
                    "frac_of_measured_hbm": round(byts / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3),
                    "kernels_per_call": kernels_per_call}
            if mode == "eager":
                line["host_us_per_call"] = round((h1 - h0) * 1e6 / calls, 2)
            print(json.dumps(line), flush=True)
        del graph
        cache.close()
        del E, WK
        torch.cuda.empty_cache()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK
    return 0


def run_profile(args):
    """A handful of launches of one kernel on the bench workload's inputs, for
    Nsight Compute: one populate (weight repack + GEMM), then two more populate
    calls, three decode steps, three alignment-weight calls, two six-layer steps of
    the cross-attention block, or a 226-step self-attention sequence (fp32)."""
    import torch
    from encoder_decoder_speech_gb300 import _build, cxa
    from encoder_decoder_speech_gb300 import workloads as W
    _build.build_library()
    cxa.load()
    torch.cuda.set_device(0)
    if args.profile in ("decode_single", "decode_single_bf16"):
        # the single-memory Whisper-Base decode (the latency-shaped kernel): populate,
        # then three decode steps
        w = W.WORKLOADS["base"]
        (E, WK, WV, bV, kl, Q, _), _ = device_inputs(torch, W, w, 0)
        cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, "bf16" if args.profile.endswith("bf16") else "f32")
        cache.populate(E, WK, WV, bV)
        for s in range(3):
            cache.decode(Q[s], kl)
        torch.cuda.synchronize()
        assert cxa.cxa_device_status(1) == cxa.CXA_OK
        return 0
    w = W.WORKLOADS[WORKLOAD]
    (E, WK, WV, bV, kl, Q, _), _ = device_inputs(torch, W, w, 0)
    bf16 = args.profile in ("decode_bf16", "shared_bf16", "shared_bf16_16")
    cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, "bf16" if bf16 else "f32")
    cache.populate(E, WK, WV, bV)
    if args.profile == "populate":
        for _ in range(2):
            cache.populate(E, WK, WV, bV)
    elif args.profile in ("shared_bf16", "shared_f32", "shared_bf16_16"):   # 8 (or 16) hypotheses per slot
        import numpy as np
        nq = 16 if args.profile == "shared_bf16_16" else 8
        Qs = torch.from_numpy(np.random.default_rng(8).standard_normal(
            (w.B, nq, w.L, w.H, w.dh)).astype(np.float32)).to("cuda")
        for _ in range(3):
            cache.decode_shared(Qs, kl)
    elif args.profile == "align":         # six alignment heads of the last three layers
        heads = [(3, 1), (4, 2), (4, 6), (5, 0), (5, 3), (5, 7)]
        for s in range(3):
            cache.alignment_weights(Q[s], kl, heads)
    elif args.profile == "block":         # two six-layer steps of the cross-attention block
        g = torch.Generator(device="cuda").manual_seed(0)

        def t(shape, std):
            return torch.randn(*shape, device="cuda", generator=g) * std

        x = t((w.B, w.d), 1.0)
        prm = [dict(WQ=t((w.d, w.d), w.d ** -0.5), WO=t((w.d, w.d), w.d ** -0.5), g=1 + t((w.d,), 0.1),
                    b=t((w.d,), 0.1), bQ=t((w.d,), 0.02), bO=t((w.d,), 0.02)) for _ in range(w.L)]
        for _ in range(2):
            for l in range(w.L):
                q = prm[l]
                cache.cross_block(l, x, q["WQ"], q["WO"], kl, ln_gamma=q["g"], ln_beta=q["b"], bQ=q["bQ"], bO=q["bO"])
    elif args.profile == "selfattn":      # the self-attention step at positions 222..225 of 448
        import numpy as np
        sa = cxa.CrossAttentionCache(w.B, 448, w.L, w.H, w.dh, "f32")
        rng = np.random.default_rng(11)
        Qs = torch.from_numpy(rng.standard_normal((4, w.B, w.L, w.H, w.dh)).astype(np.float32)).to("cuda")
        Ks = torch.from_numpy(rng.standard_normal((4, w.B, w.L, w.H, w.dh)).astype(np.float32)).to("cuda")
        out = torch.empty_like(Qs[0])
        for s in range(226):
            pos = torch.full((w.B,), s, dtype=torch.int32, device="cuda")
            sa.self_attention_step(pos, Qs[s % 4], Ks[s % 4], Ks[(s + 1) % 4], out=out)
        sa.close()
    else:
        for s in range(3):
            cache.decode(Q[s], kl)
    torch.cuda.synchronize()
    assert cxa.cxa_device_status(1) == cxa.CXA_OK
    return 0


def library_tf32_tflops(torch, n=8192, reps=10):
    """The TF32 denominator measured the way the bf16 one is: a library fp32 matmul
    of n^3 with TF32 tensor cores allowed, best of `reps` (a reference figure only;
    nothing on the product path calls it)."""
    ms = library_matmul_ms(torch, n, n, n, torch.float32, reps, best=True)
    return 2.0 * n ** 3 / (ms * 1e-3) / 1e12


def library_matmul_ms(torch, M, K, N, dtype, reps=20, best=False):
    """A library matmul [M, K] x [K, N] -> [M, N] in `dtype` (fp32 with TF32 tensor
    cores allowed), median (or best) of `reps` CUDA-event timings: the same
    contraction as a populate, without its head-major layout or bias, as a
    reference figure only (nothing on the product path calls it)."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(M, K, device="cuda", dtype=dtype)
        b = torch.randn(K, N, device="cuda", dtype=dtype)
        c = torch.empty(M, N, device="cuda", dtype=dtype)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        del a, b, c
        torch.cuda.empty_cache()
        ts.sort()
        return ts[0] if best else ts[len(ts) // 2]
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def window_psnr(torch, cxa, w, dev_inputs, oracle_path):
    """Informational parity of one whole window: the GPU's 128 decode outputs of
    the memory the oracle leg ran (populate from the packed weights, then every
    step) against the oracle's, as PSNR = 10 log10(max|ref|^2 / MSE) and max-abs.
    End to end from E (TF32 populate into an fp32 cache, then decode)."""
    import numpy as np
    E, WK, WV, bV, kl, Qs, _ = dev_inputs
    ref = np.load(oracle_path)                         # [steps, L, H, dh] of the oracle's slot
    b = 0
    cache = cxa.CrossAttentionCache(w.B, w.T, w.L, w.H, w.dh, "f32")
    packed = cache.pack_weights(WK, WV)
    cache.populate_packed(E, packed, bV)
    outs = torch.empty((w.steps, w.B, w.L, w.H, w.dh), device="cuda")
    for s in range(w.steps):
        cache.decode(Qs[s], kl, out=outs[s])
    got = outs[:, b].double().cpu().numpy()
    cache.close()
    err = got - ref
    mse = float((err ** 2).mean())
    peak = float(np.abs(ref).max())
    return {"psnr_db": 10.0 * float(np.log10(peak * peak / mse)) if mse > 0 else None,
            "max_abs": float(np.abs(err).max()), "peak_abs_ref": peak,
            "what": f"slot {b}: all {w.steps} decode steps of one window, fp32 cache, end to end from E "
                    "(TF32 populate), against the fp64 oracle; informational (the gates are in the tests)"}


def run_cxa(args):
    rank, world, local = dist_env()
    cpu_base = None
    cpu_base_mc = None
    oracle_out = None
    subsets = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle legs run first, in their own processes, before any GPU work:
        # single-threaded (its first window's outputs kept for the PSNR below), then
        # as many single-threaded processes as the host has cores, then labelled
        # subsets of the two workloads too large to run whole
        import tempfile
        fd, oracle_out = tempfile.mkstemp(prefix="oracle_window", suffix=".npy")
        os.close(fd)
        cpu_base = cpu_baseline_obj(run_oracle_subprocess(args.budget_s, args.max_slots, save_path=oracle_out))
        ncores = os.cpu_count() or 1
        if ncores > 1:
            cpu_base_mc = cpu_baseline_obj(run_oracle_subprocess(args.budget_s, args.max_slots, procs=ncores))
        subsets = {"whisper_large": run_oracle_subset_subprocess("large", args.budget_s / 2),
                   "sweep_T32768_B64": run_oracle_subset_subprocess("sweep", args.budget_s / 2)}

    import torch
    from encoder_decoder_speech_gb300 import _build, cxa
    from encoder_decoder_speech_gb300 import workloads as W

    _build.build_library()
    cxa.load()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    w = W.WORKLOADS[WORKLOAD]
    dev_inputs, host_inputs = device_inputs(torch, W, w, rank)
    kl = host_inputs[1]
    K, Wu = args.steps, args.warmup
    main = measure(torch, cxa, W, w, dev_inputs, "f32", K, Wu, rank, world, dist, timed_clocks=(rank == 0))
    variants = {}
    if not args.no_variants:
        v = measure(torch, cxa, W, w, dev_inputs, "bf16", K, Wu, rank, world, dist, timed_clocks=False)
        vb = decode_bytes(w.L, w.H, w.dh, 2, kl, w.B)
        variants["bf16_cache"] = {
            "value": world * K * w.B * w.steps / (v["total_ms"] / 1000.0), "unit": "tokens/s",
            "ms_per_step": v["total_ms"] / K,
            "decode_GBps": vb / (v["decode_launch_us"] * 1e-6) / 1e9,
            "decode_launch_us": v["decode_launch_us"], "populate_ms": v["populate_ms"]}
    e2e_ms, h2d, d2h, e2e_reps = measure_e2e(torch, cxa, w, host_inputs, dev_inputs[1:4], K, Wu, dist)
    large = None if args.no_variants else measure_populate_large(torch, cxa, W, Wu)
    tf32_lib = None if args.no_variants else library_tf32_tflops(torch)
    # the library on the populates' own contractions ([B*T, d] x [d, 2*L*d])
    lib_base_ms = None if args.no_variants else library_matmul_ms(torch, w.B * w.T, w.d, 2 * w.L * w.d,
                                                                  torch.float32)
    lib_large_ms = None if large is None else library_matmul_ms(torch, large["B"] * large["T"], large["d"],
                                                                2 * large["L"] * large["d"], torch.bfloat16)
    parity = None
    if oracle_out is not None:
        parity = window_psnr(torch, cxa, w, dev_inputs, oracle_out)
        os.unlink(oracle_out)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(local)
    tokens = world * K * w.B * w.steps
    value = tokens / (main["total_ms"] / 1000.0)
    dbytes = decode_bytes(w.L, w.H, w.dh, 4, kl, w.B)
    achieved = dbytes / (main["decode_launch_us"] * 1e-6) / 1e9
    pflops = populate_flops(w.L, w.d, w.B, w.T)
    tf32_peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * TF32_OVER_BF16
    tf32_burst = peaks["bf16_tflops"] * TF32_OVER_BF16
    pop_tflops = pflops / (main["populate_ms"] * 1e-3) / 1e12
    traffic = recorded_traffic()
    line = {
        "metric": "cross-attn decode tokens/s (batched Whisper-Base window: populate + 128 decode steps)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wu,
        "ms_per_step": main["total_ms"] / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded numpy, Whisper-Base shapes)",
        "config": dict(workload_config(w, "f32"), parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "roofline": {"bound": "hbm", "kernel": "decode_stream_kernel<f32> (persistent, last-arriver merge)",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": dbytes, "launch_us": main["decode_launch_us"],
                     "peak_source": peaks["source"], "frac_of_nominal_7900": achieved / NOMINAL_HBM_GBS},
        "populate": {"bound": "tensor", "kernel": "populate_gemm_kernel<tf32> (weights packed once)",
                     "achieved": pop_tflops, "unit": "TFLOP/s", "peak": tf32_peak,
                     "peak_note": f"{peaks['source']} bf16 sustained x 1/2 (TF32 runs at half the bf16 rate: "
                                  "4096 FLOP/clk/SM by ncu); timed inside the window loop",
                     "frac": pop_tflops / tf32_peak, "frac_of_burst": pop_tflops / tf32_burst,
                     "flops_per_call": pflops, "ms": main["populate_ms"],
                     "pack_weights_ms": main["pack_weights_ms"],
                     "library_tf32_tflops": tf32_lib,
                     "frac_of_library_tf32": None if tf32_lib is None else pop_tflops / tf32_lib,
                     "library_same_shape_ms": lib_base_ms,
                     "library_same_shape_note": "torch.matmul fp32 (TF32 allowed) of the same [B*T, d] x "
                                               "[d, 2*L*d] contraction, row-major output, no bias, median of 20",
                     "speed_vs_library_same_shape": None if lib_base_ms is None else lib_base_ms / main["populate_ms"],
                     "pack_note": "K-major repack of WK/WV, once per model load (timed apart, 10 calls)"},
        "populate_large_bf16": None if large is None else {
            "bound": "tensor", "kernel": "populate_gemm_kernel<bf16> + pack_weights",
            "workload": "whisper-large dims: 8 x E [1500,1280] bf16, 32 layers, 20x64 heads, bf16 cache",
            "achieved": large["flops_per_call"] / (large["ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
            "peak": peaks["bf16_tflops"], "peak_note": f"{peaks['source']} bf16 burst",
            "frac": large["flops_per_call"] / (large["ms"] * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "ms": large["ms"], "library_same_shape_ms": lib_large_ms,
            "speed_vs_library_same_shape": None if lib_large_ms is None else lib_large_ms / large["ms"],
            "convert_e_ms": large["convert_ms"],
            "convert_e_GBps": large["convert_bytes"] / (large["convert_ms"] * 1e-3) / 1e9,
            "convert_note": "E arrives in fp32: cxa_convert_bf16 (round to nearest even) before each populate, "
                            "timed apart; weights converted and packed once"},
        "decode_large_bf16": None if large is None else {
            "bound": "hbm", "kernel": "decode_stream_kernel<bf16>",
            "workload": "whisper-large dims: 8 memories x 1500 keys, 32 layers, 20x64 heads, bf16 cache, "
                        f"{large['steps']} steps, fresh queries each",
            "us_per_step": large["decode_us"], "tokens_per_s": large["B"] / (large["decode_us"] * 1e-6),
            "achieved": large["decode_bytes"] / (large["decode_us"] * 1e-6) / 1e9, "unit": "GB/s",
            "peak": peaks["hbm_gbs"],
            "frac": large["decode_bytes"] / (large["decode_us"] * 1e-6) / 1e9 / peaks["hbm_gbs"]},
        "clocks": main["clocks"],
        "spread_ms": main["spread_ms"],
        "e2e": {"value": tokens / (e2e_ms / 1000.0), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "note": "E, key_len and 128 Q copied in, 128 outputs copied out per "
                                                     "window from/to pinned host memory on a copy stream that "
                                                     "double-buffers against the compute stream; weights resident; "
                                                     "median of three timed runs of the K windows",
                "runs_tokens_per_s": [round(tokens / (m / 1000.0), 1) for m in e2e_reps]},
        "gpu_launches": main["launches"],
        "variants": variants,
        "device": {"name": props.name, "sms": props.multi_processor_count,
                   "lib_sha": source_sha([os.path.join(ROOT, "encoder_decoder_speech_gb300", "_lib", "libcxa.so")])},
    }
    if parity is not None:
        line["parity"] = parity
    line["provenance"] = provenance()
    if cpu_base is not None:
        line["cpu_baseline"] = cpu_base
    if subsets is not None:
        line["cpu_baseline_subsets"] = subsets
    if cpu_base_mc is not None:
        line["cpu_baseline_multicore"] = cpu_base_mc
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_subset:
        print(json.dumps(oracle_subset(args.oracle_subset, args.budget_s)))
        return 0
    if args.oracle_small:
        print(json.dumps(oracle_small_window(args.oracle_small)))
        return 0
    if args.oracle_sample:
        if args.procs > 1:
            print(json.dumps(oracle_sample_procs(args.budget_s, args.max_slots, args.procs)))
        else:
            print(json.dumps(oracle_sample(args.budget_s, args.max_slots, args.warmup, save_path=args.save)))
        return 0
    if args.profile:
        return run_profile(args)
    if args.sweep:
        return run_sweep(args)
    if args.shared:
        return run_shared(args)
    if args.small:
        return run_small(args)
    if args.block:
        return run_block(args)
    if args.selfattn:
        return run_selfattn(args)
    if args.align:
        return run_align(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_cxa(args)


if __name__ == "__main__":
    sys.exit(main())
