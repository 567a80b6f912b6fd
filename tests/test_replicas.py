"""The multi-GPU path is replicas: one process per GPU, each streaming its own
videos, with the max over ranks of the timed region as the job's time.  Its
host logic runs here as two gloo ranks on the CPU (no GPU involved)."""

from __future__ import annotations

import argparse
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


def _rank_main(rank: int, world: int, port: int, root: str, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, root)
    import bench
    from synth import SHAPES, FrameSource
    dist, r, ws, local = bench._dist()
    sh = SHAPES["tiny_f32"]
    q0 = FrameSource(sh, seed=bench.replica_seed(sh, r)).frame(0)[0]
    slowest = bench.max_over_ranks(1.5 + r, dist)           # rank r "took" 1.5 + r
    dist.barrier()
    q.put((r, ws, local, slowest, bench.replica_seed(sh, r), float(q0.sum())))
    dist.destroy_process_group()


def test_two_replicas_share_only_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, ROOT, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    assert [g[:3] for g in got] == [(0, 2, 0), (1, 2, 1)]
    assert all(g[3] == 2.5 for g in got)                  # both see the slower rank's time
    assert got[0][4] != got[1][4] and got[0][5] != got[1][5]   # independent streams


def test_reference_arm_is_rank0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from synth import SHAPES
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=1, warmup=0, gpus=2)
    bench.run_reference(args, SHAPES["internvl3_2b_stack"])   # returns at once on rank 1
    assert capsys.readouterr().out == ""


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, None) == 3.25
