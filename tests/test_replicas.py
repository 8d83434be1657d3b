"""The N>1 path of the benchmark (CPU, gloo, world_size 2): replicas only.

The attention path shards into independent (sequence, kv head) problems, so
under torchrun every rank runs its own replica and the only collective is
the max over ranks of the timed region.  This runs that host logic with two
gloo ranks on the CPU.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_info()
        assert (w, r, l) == (world, rank, rank)
        ms = 10.0 + 5.0 * rank                 # the ranks' own times differ
        dist.barrier()
        job_ms = bench.max_over_ranks(ms, world)
        out[rank] = (job_ms, bench.job_throughput(1e12, job_ms, world))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_whole_job_rate():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0
    # 2 replicas x 1 TFLOP each in 15 ms
    assert abs(out[0][1] - 2 * 1e12 / 15e-3 / 1e12) < 1e-9


def test_single_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1e12, 1.0, 1) == 1000.0
