"""The bench's multi-GPU path on CPU: N independent replicas, no data exchange; the job's time is
the slowest rank's and its throughput counts the units of every rank. Two gloo ranks stand in for
two GPUs."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 1 + r seconds for the timed steps and 3 - r for the end-to-end ones
        el, e2e = bench.max_over_ranks([1.0 + rank, 3.0 - rank])
        q.put((rank, el, e2e, bench.replica_throughput(world, 524292, 10, el)))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_sum_the_units():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(120)
        assert pr.exitcode == 0
    got = sorted(q.get() for _ in range(world))
    for rank, el, e2e, value in got:
        assert el == 2.0 and e2e == 3.0          # max over ranks, on every rank
        assert value == 2 * 524292 * 10 / 2.0    # both ranks' tokens over the slowest time


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.replica_throughput(1, 100, 3, 2.0) == 150.0
