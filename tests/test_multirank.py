"""The bench's multi-GPU path, run as two gloo ranks on the CPU.

The path shards only as replicas: N independent copies of the step with no
data-path collective.  What crosses ranks is the timing: a barrier on both sides
of the timed region, the maximum time over ranks, and the whole-job throughput
(every replica's work over the slowest replica's time).
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    bench.barrier(world)
    local_ms = 100.0 + 25.0 * rank                      # rank 1 is the slowest replica
    mx = bench.max_over_ranks(world, local_ms)
    value = bench.whole_job_tflops(world, 1.0e12, 10, mx)
    bench.barrier(world)
    out[rank] = (mx, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_time_as_the_slowest_replica():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        mx, value = out[r]
        assert mx == 125.0
        assert value == pytest.approx(2 * 1.0e12 * 10 / 0.125 / 1e12)


def test_single_rank_helpers():
    import bench

    assert bench.max_over_ranks(1, 3.5) == 3.5
    assert bench.whole_job_tflops(1, 2.0e12, 5, 1000.0) == pytest.approx(10.0)
