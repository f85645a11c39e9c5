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


def _shard_worker(rank, world, port, total, q):
    """One rank: verify its row block with the oracle (the CUDA path's
    stand-in on a CPU rank), row_base = the block's first row, then gather."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    from oracle import verify as ov
    from speculative_decoding_verify_07_gb300 import binding as sv
    from speculative_decoding_verify_07_gb300 import synth
    inp = synth.make_mixed(B=total, k=2, V=2048, seed_offset=5)
    lo, hi = sv.row_block(total, world, rank)
    part = ov.verify(inp.logits[lo:hi], inp.q[lo:hi], inp.drafts[lo:hi], inp.temperature[lo:hi],
                     inp.top_k[lo:hi], inp.top_p[lo:hi], inp.seed, row_base=lo)
    mine = {k_: part[k_] for k_ in ("tokens", "accept_len", "logprobs", "alpha", "flags")}
    parts = [None] * world
    dist.all_gather_object(parts, (lo, hi, mine))
    if rank == 0:
        q.put(parts)
    dist.destroy_process_group()


@pytest.mark.parametrize("total", [8, 7])
def test_row_blocks_over_two_gloo_ranks_equal_one_call(total):
    """Rows split over 2 ranks, each verifying its block with row_base = its
    first row, give exactly the outputs of verifying the whole batch at once
    (every row draws the random numbers of its place in the batch)."""
    import numpy as np
    from oracle import verify as ov
    from speculative_decoding_verify_07_gb300 import synth
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_shard_worker, args=(2, _free_port(), total, q), nprocs=2, join=True,
                       start_method="spawn")
    parts = q.get()
    blocks = [(lo, hi) for lo, hi, _ in parts]
    assert blocks[0][0] == 0 and blocks[-1][1] == total
    assert all(blocks[i][1] == blocks[i + 1][0] for i in range(len(blocks) - 1))
    inp = synth.make_mixed(B=total, k=2, V=2048, seed_offset=5)
    full = ov.verify(inp.logits, inp.q, inp.drafts, inp.temperature, inp.top_k, inp.top_p, inp.seed)
    for key in ("tokens", "accept_len", "logprobs", "alpha", "flags"):
        joined = np.concatenate([p[key] for _, _, p in parts])
        assert np.array_equal(joined, full[key]), key
    # the shards are not trivially equal: a row's draws depend on its place
    shifted = ov.verify(inp.logits[1:], inp.q[1:], inp.drafts[1:], inp.temperature[1:], inp.top_k[1:],
                        inp.top_p[1:], inp.seed, row_base=0)
    assert not all(np.array_equal(shifted[k_], full[k_][1:]) for k_ in ("tokens", "accept_len"))


def test_row_block_partition():
    from speculative_decoding_verify_07_gb300 import binding as sv
    for total in (0, 1, 7, 64, 129):
        for world in (1, 2, 3, 8):
            spans = [sv.row_block(total, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == total
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
    with pytest.raises(ValueError):
        sv.row_block(8, 2, 2)
