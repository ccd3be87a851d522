"""The benchmark's multi-rank path on CPU: two gloo ranks, each an independent replica; the
job's clock is the slowest rank and its throughput counts the units of every rank."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.aggregate(10.0 * (rank + 1), 1024, 5, world, "cpu")
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value in res:
        assert ms == 20.0                                   # the slower rank's time, on every rank
        assert value == pytest.approx(2 * 1024 * 5 / 0.020)  # units of both ranks / slowest time


def test_aggregate_single_rank():
    import bench
    ms, value = bench.aggregate(4.0, 100, 10, 1, "cpu")
    assert ms == 4.0 and value == pytest.approx(100 * 10 / 0.004)
