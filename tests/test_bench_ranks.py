"""Host logic of bench.py's multi-rank runs, on the CPU with two gloo ranks.

Under torchrun every rank runs an independent replica of the layer; the job's
time is the slowest rank's, and the job's throughput counts every rank's
tokens.  The reference arm runs on rank 0 alone.  These tests drive the same
helpers bench.py uses, with the gloo backend instead of NCCL.
"""

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        secs = 0.5 + rank  # rank 1 is the slower one
        slowest = bench.max_over_ranks(secs, world)
        value = bench.job_throughput(64 * 100, world, slowest)
        # the reference arm prints on rank 0 only; other ranks return at once
        args = type("A", (), {"tokens": 1})()
        ran = bench.run_reference(args, None, world, rank) if rank != 0 else "skipped"
        out.put((rank, slowest, value, ran))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, value, ran in got:
        assert slowest == pytest.approx(1.5)          # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 6400 / 1.5)  # both ranks' tokens over the slowest time
    assert got[1][3] is None                           # rank 1 did no reference work


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks(0.25, 1) == 0.25
    assert bench.job_throughput(6400, 1, 0.5) == pytest.approx(12800)
