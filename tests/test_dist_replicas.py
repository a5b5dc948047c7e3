"""Replica plumbing on CPU: two gloo ranks join through the same helpers the
benchmark uses, meet at a barrier and agree on the max and sum of per-rank
values (the benchmark's max-over-ranks step time and whole-job work)."""
import os
import socket

import torch.multiprocessing as mp

from fp8_block_scaled_16_b300 import dist as D


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    r = D.init_from_env("gloo")
    try:
        assert r.initialized and r.world == world and r.rank == rank
        D.barrier(r)
        mx = D.max_over_ranks(r, 10.0 + rank)
        sm = D.sum_over_ranks(r, 1.5 * (rank + 1))
        D.barrier(r)
        q.put((rank, mx, sm))
    finally:
        D.shutdown(r)


def test_two_gloo_replicas_agree_on_max_and_sum():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 11.0, 4.5), (1, 11.0, 4.5)]


def test_single_process_is_a_no_op():
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    r = D.init_from_env("gloo")
    assert not r.initialized and r.world == 1
    D.barrier(r)
    assert D.max_over_ranks(r, 3.0) == 3.0 and D.sum_over_ranks(r, 3.0) == 3.0
