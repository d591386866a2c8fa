"""The benchmark's multi-rank path on CPU (gloo, world size 2): every rank
runs its own replica, the reported time is the maximum over ranks, and rank 0
alone prints.  No GPU and no data-path collective are involved."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    env = bench.dist_env()
    t = bench.max_over_ranks(10.0 * (rank + 1), ws)
    bench.barrier(ws)
    results[rank] = (env, t)
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ws = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, ws, port, results)) for r in range(ws)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        got = dict(results)
    assert got[0][0] == (2, 0, 0) and got[1][0] == (2, 1, 1)
    assert got[0][1] == got[1][1] == 20.0


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0"])
    assert capsys.readouterr().out == ""
