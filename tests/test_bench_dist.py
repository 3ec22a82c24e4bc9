"""bench.py's multi-rank aggregation (barrier + max over ranks) with two gloo
processes on the CPU.  Replicas do not exchange data; only the timing is
reduced."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_env()
        assert (w, r, l) == (world, rank, rank)
        bench.barrier(world)
        slowest = bench.reduce_max(1.5 + rank, world)
        q.put((rank, slowest))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_single_process_reduce_is_identity():
    import bench

    assert bench.reduce_max(3.25, 1) == 3.25


def test_live_copy_pieces_cover_exactly_the_live_rows():
    """The end-to-end step's copy list: q and the lengths whole, and rows
    [0, L_b) of every sequence's K and V (empty sequences copy nothing).
    Copying it onto a poisoned destination leaves exactly the rows past
    each length poisoned."""
    import torch

    import bench

    B, cap, Hkv, d, lens = 4, 37, 2, 8, [37, 0, 5, 19]
    src = (torch.randn(B, 1, 4, d), torch.randn(B, cap, Hkv, d), torch.randn(B, cap, Hkv, d),
           torch.tensor(lens, dtype=torch.int32))
    dst = tuple(torch.full_like(x, -7) for x in src)
    pieces = bench.live_copy_pieces(dst, src, lens)
    assert len(pieces) == 2 + 2 * sum(1 for n in lens if n > 0)
    for a, b in pieces:
        a.copy_(b)
    assert torch.equal(dst[0], src[0]) and torch.equal(dst[3], src[3])
    for c in (1, 2):
        for b, n in enumerate(lens):
            assert torch.equal(dst[c][b, :n], src[c][b, :n])
            assert bool((dst[c][b, n:] == -7).all())
    moved = sum(s.numel() * s.element_size() for _, s in pieces)
    assert moved == (src[0].numel() + 2 * sum(lens) * Hkv * d) * 4 + 4 * B
