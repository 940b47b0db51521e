"""Replica aggregation of bench.py on CPU: two gloo ranks, max-over-ranks time and job throughput."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    got = bench.max_over_ranks(ms, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 15.0


def test_job_throughput_counts_every_rank_over_the_slowest_time():
    import bench
    # two ranks, 1e12 flop each, slowest 10 ms -> 2e12 / 0.01 s
    assert bench.job_throughput(1e12, 2, 10.0) == pytest.approx(2e14)
    assert bench.job_throughput(5e11, 1, 1.0) == pytest.approx(5e14)
