"""The N > 1 bench path on CPU: two gloo ranks as replicas.

bench.py runs one replica of the GEMM per GPU with no collective on the data
path; the ranks only meet at a barrier around the timed region and in one MAX
reduction of their times, and rank 0 reports the units of all ranks over the
slowest rank's time. Those host steps are exercised here with world size 2 on
the gloo backend (no GPU).
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.init_dist(world, backend="gloo")
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    ms_max = bench.max_over_ranks(ms, w)
    value = bench.job_throughput(100.0, w, ms_max)
    results[rank] = (ms_max, value)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_replicas_reduce_with_max_and_sum_units():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1] == (15.0, 2 * 100.0 / 15.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(7.0, 1, 2.0) == 3.5
