"""Host logic of bench.py's multi-rank path on CPU: world_size 2 over gloo.

Under torchrun every rank runs an independent replica of the one-GPU workload
(weak scaling, no data-path collective); the only cross-rank step is taking the
slowest rank's time, and the reported value is the work of all ranks over that
time.  The reference arm prints from rank 0 only.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], dist)
        out[rank] = (slowest, bench.whole_job_tflops(10 ** 12, world, 5, slowest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    times = [120.0, 150.0]  # ms for 5 steps of 1 TFLOP each, per rank
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    # 2 ranks x 5 steps x 1 TFLOP over the slowest 0.150 s
    assert abs(res[0][1] - 2 * 5 / 0.150) < 1e-9
    assert res[0][1] == res[1][1]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert abs(bench.whole_job_tflops(2 * 10 ** 12, 1, 10, 1000.0) - 20.0) < 1e-12


def test_reference_arm_prints_from_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        cpu_workers, cpu_rows, warmup, steps = 1, 8, 3, 1

    assert bench.bench_reference(A, rank=1, world=2) is None
