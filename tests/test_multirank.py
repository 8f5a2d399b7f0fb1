"""The bench's multi-rank path on CPU: world size 2 over gloo.

Replicas run independently (the path shards with no exchange step); the only
collective is the max over ranks of the timings, and the whole-job GB/s counts
every rank's bytes over the slowest rank's time.  The reference arm prints on
rank 0 only.
"""
import io
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out = bench.max_over_ranks([1.5 + rank, 10.0 - 3 * rank], world, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out))


def test_timings_take_the_slowest_rank_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.5, 10.0]


def test_single_rank_is_identity_and_job_bandwidth_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1, None) == [3.0, 4.0]
    one = bench.job_gbps(672_202_752, 166.0, 1)
    assert abs(one - 672_202_752 / 166e-6 / 1e9) < 1e-9
    assert abs(bench.job_gbps(672_202_752, 166.0, 4) - 4 * one) < 1e-9


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import synth
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "gpus": 2})(), synth.WORKLOADS["tiny_8k_g4_d64"])
    assert buf.getvalue() == ""
