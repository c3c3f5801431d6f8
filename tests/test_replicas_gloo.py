"""The multi-GPU path of the benchmark is independent replicas (no data-path collective):
every rank runs the whole workload on its own GPU, and rank 0 reports the KV bytes of all
ranks over the slowest rank's time.  This checks that aggregation with two gloo ranks on
the CPU, and that the reference arm leaves ranks other than 0 idle."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [10.0 + 5.0 * rank, 20.0 - 3.0 * rank]        # rank 1 is slower on the first
        q.put((rank, bench.slowest_rank(ms, torch.device("cpu"))))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_job_rate_with_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got[0] == got[1] == [15.0, 20.0]
    sys.path.insert(0, ROOT)
    import bench
    # two replicas of 286.72 MB in 200 calls over the slowest rank's 11.0 ms
    assert bench.job_tbs(286_720_000, 2, 200, 11.0) == pytest.approx(2 * 286.72e6 * 200 / 11e-3 / 1e12)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    bench.run_reference(bench.parse_args())                      # returns at once: no oracle work on rank 1
    assert capsys.readouterr().out == ""
