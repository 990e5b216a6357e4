"""bench.py's N > 1 rules on CPU: each rank is an independent replica, the
job's time is the slowest rank's (element-wise max over ranks, as bench.py
all-reduces it), and the throughput counts all ranks' FLOPs.  Two gloo ranks
on 127.0.0.1."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (10 + r) ms in total and a (2 - r) ms GEMM average
        local = [10.0 + rank, 2.0 - rank]
        tot, gemm = bench.max_over_ranks(local, dist, "cpu")
        value = bench.replica_throughput(world, 1e12, 100, tot)
        out.put((rank, tot, gemm, value))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tot, gemm, value in res:
        assert tot == 11.0 and gemm == 2.0           # max over ranks, element-wise
        # 2 replicas x 100 steps x 1e12 FLOP in 11 ms
        assert value == pytest.approx(2 * 100 * 1e12 / 11e-3 / 1e12)


def test_single_replica_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 4.5], None, "cpu") == [3.0, 4.5]
    assert bench.replica_throughput(1, 2e12, 10, 20.0) == pytest.approx(1000.0)
