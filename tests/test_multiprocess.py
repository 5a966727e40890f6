"""The multi-GPU path of the benchmark, on the CPU with gloo (world size 2).

The compressor shards by tensor with no exchange, so N GPUs run N
independent replicas (bench.py --gpus N under torch.distributed.run). The
only cross-rank logic is the timing: every rank's times are reduced to the
slowest rank's, and the job's throughput counts the units of all ranks over
that time. This runs that logic as two gloo processes.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local = [1.0 + rank, 5.0 - rank, 0.25 * rank]
        q.put((rank, bench.max_over_ranks(local, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = dict(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    # the slowest rank's value of every timing, on both ranks
    assert results[0] == results[1] == [2.0, 5.0, 0.25]


def test_single_process_values_pass_through():
    import bench
    assert bench.max_over_ranks([3.0, 1.5], "cpu") == [3.0, 1.5]


@pytest.mark.parametrize("world", [1, 2, 8])
def test_replica_value_counts_every_rank(world):
    import bench
    # each rank processed 1 GB per step for 10 steps; the slowest took 4 s
    assert bench.replica_value(1e9, 10, world, 4.0) == pytest.approx(world * 2.5e9)
