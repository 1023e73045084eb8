"""The benchmark's multi-rank host logic on CPU with gloo, world size 2:
replicas draw different data, the timing is the max over ranks, and the
whole-job value counts every rank's bytes."""

import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank
        mx = bench.max_over_ranks(local_ms, dist, "cpu")
        seeds = [bench.replica_seed(s, rank) for s in (0, 1, 2, 3)]
        dist.barrier()
        q.put((rank, mx, seeds))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_seeds():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[1] for o in out] == [15.0, 15.0]
    assert set(out[0][2]).isdisjoint(out[1][2])


def test_whole_job_value_counts_every_rank():
    assert bench.whole_job_gbs(10**9, 10, 1, 1000.0) == pytest.approx(10.0)
    assert bench.whole_job_gbs(10**9, 10, 4, 1000.0) == pytest.approx(40.0)
    assert bench.max_over_ranks(3.0, None) == 3.0


def test_replica_inputs_differ_between_ranks():
    from fp8_communication_compression_gb300 import workloads as W

    a = W.tp_activation(bench.replica_seed(0, 0), 4, 256)
    b = W.tp_activation(bench.replica_seed(0, 1), 4, 256)
    assert not np.array_equal(a, b)
