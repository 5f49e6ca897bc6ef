"""The replica path of bench.py with two ranks on CPU (gloo): every rank
voxelizes its own frames, the timed region is the maximum over ranks, the
whole-job rate counts every rank's points, and the reference arm runs and
prints on rank 0 only.  No GPU and no collective on the data path."""

from __future__ import annotations

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        region = 10.0 + 5.0 * rank  # rank 1 is the slow one
        worst = bench.max_over_ranks(region)
        args = type("A", (), {"workload": "tiny", "steps": 2, "warmup": 1, "gpus": world, "batch": 1, "op": "voxelize"})()
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(args, rank, world)
        q.put((rank, worst, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [15.0, 15.0]       # both ranks see the slowest rank's time
    assert '"impl": "reference"' in got[0][2]         # rank 0 prints the reference line
    assert got[1][2] == ""                            # other ranks do no work and print nothing


def test_whole_job_rate_counts_every_rank():
    one = bench.whole_job_rate(122_880, 100, 1, 3.0)
    four = bench.whole_job_rate(122_880, 100, 4, 3.0)
    assert four == pytest.approx(4 * one)
    assert one == pytest.approx(122_880 * 100 / 3e-3 / 1e6)


def test_max_over_ranks_without_group_is_identity():
    assert bench.max_over_ranks(7.5) == 7.5
