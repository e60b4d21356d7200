"""The benchmark's multi-rank plumbing (replicas: one independent decode step
per GPU, max time over ranks, rank 0 prints), run as two gloo ranks on the CPU:
no GPU is involved."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import io
    import contextlib

    import bench
    dist, r, w, local = bench.dist_setup(world)
    # rank r took (r + 1) seconds: the job's time is the slowest rank's
    t = bench.max_over_ranks(dist, float(r + 1), "cpu")
    bench.barrier(dist)
    # the reference arm under N > 1: rank 0 alone runs it, the others return
    # at once and print nothing
    printed = io.StringIO()
    if r != 0:
        with contextlib.redirect_stdout(printed):
            bench.bench_reference(type("A", (), {"steps": 1, "warmup": 0})())
    out.put((r, w, local, t, printed.getvalue()))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_max_over_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=100) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    assert all(r[1] == world and r[2] == r[0] for r in results)
    assert all(r[3] == 2.0 for r in results)   # the max of 1.0 and 2.0, on every rank
    assert results[1][4] == ""                  # a non-zero rank prints no reference line


def test_replica_value_is_whole_job_throughput():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas, 100 steps each, slowest rank 0.05 s: 4000 steps/s for the job
    assert bench.replica_throughput(world=2, steps=100, t_max=0.05) == pytest.approx(4000.0)
