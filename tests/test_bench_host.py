"""Host logic of the benchmark's multi-rank (replica) mode on CPU with gloo,
world size 2: the maximum over ranks and the whole-job aggregate."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(10.0 + rank)  # rank 1 is slower
    value = bench.replica_throughput(tokens_per_step=1000, steps=5, world=world, ms=slowest)
    q.put((rank, slowest, value))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slowest, value in got:
        assert slowest == 11.0
        assert value == pytest.approx(world * 5 * 1000 / 0.011)


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5  # no process group: identity
    assert bench.replica_throughput(100, 2, 1, 1000.0) == pytest.approx(200.0)
