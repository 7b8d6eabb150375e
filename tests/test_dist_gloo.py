"""The benchmark's multi-rank host logic on CPU: two gloo ranks.

With N GPUs every rank runs the same workload on its own device (replicas, no
data-path collective); the timed region is bracketed by barriers, the step
time is the max over ranks and the work is the sum over ranks.  This checks
that reduction on CPU with world_size 2.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist = bench.init_dist(world, "gloo")
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower one
    local_units = 1000 * (rank + 1)
    ms, units = bench.combine_ranks(local_ms, local_units, world, "cpu")
    bench.barrier(world)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_two_rank_max_time_sum_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, units in got:
        assert ms == 15.0            # max over ranks
        assert units == 3000.0       # sum over ranks


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 1
    bench.bench_reference(A())
    assert capsys.readouterr().out == ""
