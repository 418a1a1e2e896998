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


def test_profile_summaries_carry_traffic_and_source_hash():
    """Every ncu summary the benchmark reads a traffic figure from exists, gives the figure and the
    hash of the kernel sources it was taken on, and names only committed files in its command; the
    sources it hashes exist. (Whether the hash matches the current sources decides whether the
    benchmark reports the figure or null; that is not asserted here.)"""
    import re
    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    names = set(re.findall(r'kernel_traffic\("(\w+)", (?:args\.case|(\d+)|"(\w+)")\)',
                           open(os.path.join(root, "bench.py")).read()))
    assert names, "no profile lookups found in bench.py"
    for kernel, num, label in names:
        for name in ([f"{kernel}_case{c}.md" for c in (1, 2, 3)] if not (num or label)
                     else [f"{kernel}_case{num}.md" if num else f"{kernel}_{label}.md"]):
            text = open(os.path.join(root, "profiles", name)).read()
            assert re.search(r"traffic_bytes_per_launch:\s*[0-9.eE+]+", text), name
            assert re.search(r"source_sha256:\s*[0-9a-f]{64}", text), name
            assert "_work/" not in text, name
        for src in bench.KERNEL_SOURCES[kernel]:
            assert os.path.exists(os.path.join(root, "rl_post_loss_gb300", "csrc", src)), src
