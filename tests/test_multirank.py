"""The multi-rank host logic of bench.py on CPU with two gloo ranks: the
max-over-ranks timing, the whole-job throughput, and which rank reports.
(The data path has no collective: each rank runs its own shard.)"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max(10.0 * (rank + 1), dist, torch.device("cpu"))
        v = bench.job_tflops(1e12, world, 4, t)
        out[rank] = (t, v)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_job_throughput():
    world, port = 2, free_port()
    out = mp.Manager().dict()
    mp.spawn(worker, args=(world, port, out), nprocs=world, join=True)
    # both ranks see the slowest rank's time (20 ms) and the same whole-job value
    assert out[0][0] == out[1][0] == 20.0
    assert out[0][1] == out[1][1] == pytest.approx(2 * 1e12 * 4 / 0.020 / 1e12)


def test_single_rank_helpers_without_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, None, None) == 3.5
    assert bench.job_tflops(2e12, 1, 10, 1000.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    from attention_forward_06_gb300.inputs import WORKLOADS

    class A:
        steps, warmup = 1, 0

    assert bench.run_reference(A, WORKLOADS["tiny"], rank=1, world=2) is None
    line = bench.run_reference(A, WORKLOADS["tiny"], rank=0, world=2)
    assert line["impl"] == "reference" and line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
