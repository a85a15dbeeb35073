"""Replica aggregation of bench.py across ranks, on CPU with gloo at world
size 2: the step time every rank reports is the maximum over ranks, the
whole-job value counts the work of all ranks, and the reference arm does its
work on rank 0 only."""
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


def _worker(rank: int, ws: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench._dist()
        ms = [3.0, 5.0][rank]                      # rank 1 is the slower replica
        mx = bench._barrier_max(ms, got_ws, torch.device("cpu"))
        value = bench._replica_throughput(1e12, mx, got_ws)
        # the reference arm returns at once on every rank but 0
        ref = bench.run_reference(None, got_ws, got_rank, got_local) if rank != 0 else "skipped"
        out.put((rank, got_ws, got_rank, mx, value, ref))
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_world_size_2():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(out.get(timeout=5) for _ in range(2))
    for rank, ws, got_rank, mx, value, ref in res:
        assert ws == 2 and got_rank == rank
        assert mx == 5.0                            # max over ranks, seen by both
        # 2 replicas x 1e12 FLOP each in 5 ms = 400 TFLOP/s whole-job
        assert value == pytest.approx(400.0)
    assert res[1][5] is None                        # rank 1: no reference work


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._barrier_max(7.5, 1, torch.device("cpu")) == 7.5
    assert bench._replica_throughput(2e12, 10.0, 1) == pytest.approx(200.0)
