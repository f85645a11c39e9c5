"""Multi-process host logic of the benchmark, on CPU with the gloo backend.

The verify path shards by rows with no exchange; the only cross-rank steps
are the timing barrier and the max-over-ranks of the elapsed time, and the
job throughput counts the rows of every rank.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [0.5, 0.8][rank]
    slowest = bench.max_over_ranks(elapsed, world, device="cpu")
    bench.barrier(world)
    rows = bench.job_rows_per_s(64 * 10, world, slowest)
    q.put((rank, slowest, rows))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_rows():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, q), nprocs=2, join=True, start_method="spawn")
    got = sorted(q.get() for _ in range(2))
    for rank, slowest, rows in got:
        assert slowest == pytest.approx(0.8)
        assert rows == pytest.approx(64 * 10 * 2 / 0.8)
