"""bench.py's multi-rank harness on CPU: two gloo ranks agree on the max of
their timings, as the weak-scaling replicas do under torchrun."""
from __future__ import annotations

import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench

    r, ws, _ = bench.dist_setup()
    assert (r, ws) == (rank, world)
    bench.barrier(ws)
    out[rank] = bench.max_over_ranks(1.5 + rank, ws)
    torch.distributed.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}
