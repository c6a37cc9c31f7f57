"""Multi-process host logic of bench.py on CPU (gloo, world size 2): the
replicas' timings are combined by max over ranks, and the whole-job
throughput counts every rank's tokens over the slowest rank's time."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 1.0 + rank * 0.5          # rank 1 is the slower replica
        m = bench.max_over_ranks(local)
        v = bench.replica_throughput(world, 2, 100, m)
        q.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_replica_timing_is_max_over_ranks_and_throughput_counts_all_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in res:
        assert m == pytest.approx(1.5)
        assert v == pytest.approx(2 * 2 * 100 / 1.5)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.replica_throughput(1, 1, 10, 2.0) == 5.0
