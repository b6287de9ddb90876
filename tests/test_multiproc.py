"""Multi-process host logic of the benchmark on CPU (gloo, world size 2): each rank
owns distinct encoder memories (weak scaling, no data-path collective) and the
job time is the maximum over ranks."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from encoder_decoder_speech_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slots = bench.rank_slots(rank, 16)
        gathered = [None] * world
        dist.all_gather_object(gathered, slots)
        t = bench.max_over_ranks(dist, [10.0 + rank, 5.0 - rank], "cpu")
        q.put((rank, gathered, t))
    finally:
        dist.destroy_process_group()


def test_two_ranks_own_distinct_memories_and_take_the_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, gathered, t in res:
        assert t == [11.0, 5.0]
        all_slots = [s for g in gathered for s in g]
        assert len(all_slots) == len(set(all_slots)) == 32
    w = W.WORKLOADS["batched_base"]
    flat = W.replace(w, ragged=False)
    assert not np.array_equal(W.make_E(flat, 0)[:4], W.make_E(flat, 16)[:4])


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
