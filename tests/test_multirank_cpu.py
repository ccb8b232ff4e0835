"""bench.py's multi-rank accounting on two gloo ranks (CPU): every rank sees
the slowest rank's time, and throughput counts every rank's tokens (weak
scaling, one independent batch per rank, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [120.0, 180.0][rank]
    got = bench.max_over_ranks(ms, world, device="cpu")
    value = bench.job_throughput(world, 16384, 20, got)
    bench.barrier(world)
    q.put((rank, got, value))
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [180.0, 180.0]
    assert res[0][2] == pytest.approx(2 * 16384 * 20 / 0.18)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(1, 100, 10, 1000.0) == pytest.approx(1000.0)
