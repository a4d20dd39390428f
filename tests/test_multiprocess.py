"""The multi-process host logic of bench.py (replicas only: no collective on the
data path) on two CPU ranks over gloo.  Each rank would run its own replica of the
workload; what the ranks share is the timing barrier, the max over ranks and the
rank-0-only report, and that is what these tests run."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # every rank gets the slowest rank's step time
        ms = bench.max_over_ranks(1.0 + rank, world)
        rate = bench.aggregate_rate(8192, ms, world)
        bench.barrier(world)
        # the reference arm: rank 0 alone runs and prints; the others return at once
        args = type("A", (), {"warmup": 0, "steps": 1, "gpus": world})()
        buf = io.StringIO()
        if rank != 0:
            with redirect_stdout(buf):
                bench.run_reference(args, world, rank)
        out_q.put((rank, ms, rate, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, printed in results:
        assert ms == 2.0                           # max over ranks, on every rank
        assert rate == pytest.approx(2 * 8192 / 2e-3)  # whole-job tokens/s at the slowest rank's pace
        if rank != 0:
            assert printed == ""                   # non-zero ranks print nothing


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_rate(100, 10.0, 1) == pytest.approx(1e4)
