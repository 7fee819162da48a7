"""Replica logic of bench.py on CPU: world_size 2 over gloo.

The path shards by request with no collective on the data path; the only
cross-rank steps are the barrier and the max-over-ranks timing.  These tests
run two ranks as processes on the CPU and check that the job throughput is
computed from the slowest rank and counts every rank's units, and that each
replica draws a different batch.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    bench.barrier(world)
    ms = bench.max_over_ranks(times[rank], world)
    value = bench.job_throughput(1280, ms, world)
    w = workloads.WORKLOADS["tiny"]
    inp = workloads.make_inputs(w, seed=bench.replica_seed(w, rank), with_target_noise=False)
    out[rank] = (ms, value, float(inp["h"].float().sum()))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_all_units():
    world, port = 2, _free_port()
    times = [2.5, 4.0]  # ms per step measured by each rank
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 4.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1280 / 4.0e-3)
    assert res[0][2] != res[1][2]  # independent batches per replica


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(1280, 2.0, 1) == pytest.approx(640000.0)
