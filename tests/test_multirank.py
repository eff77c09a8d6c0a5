"""The N > 1 plumbing of bench.py, exercised with two gloo ranks on the CPU.

The benchmark shards by replication (every rank runs its own copy of the workload, no data-path
collective); the only cross-rank operations are the barrier around the timed region and the max over
ranks of the step time.  These tests run them as two processes on 127.0.0.1.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    w, r, local = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    # each rank "measured" a different step time; the job is timed by the slowest rank
    ms = 1.5 + rank
    slowest = bench.max_over_ranks(ms, w)
    value = bench.whole_job_value(8192, w, slowest / 1e3)
    bench.barrier(w)
    out.put((r, w, local, slowest, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert [r[0] for r in res] == [0, 1]
    for rank, w, local, slowest, value in res:
        assert w == world and local == rank
        assert slowest == pytest.approx(2.5)  # max over ranks, identical on every rank
        assert value == pytest.approx(8192 * world / 2.5e-3)  # weak scaling: all ranks' units / slowest time


def _reference_rank(rank: int, world: int, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, world

    bench.run_reference(Args)  # returns at once on ranks other than 0
    out.put(rank)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun only rank 0 times the oracle; the other ranks exit without work."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_reference_rank, args=(1, 2, q))
    p.start()
    p.join(timeout=60)
    assert p.exitcode == 0
    assert q.get(timeout=5) == 1
