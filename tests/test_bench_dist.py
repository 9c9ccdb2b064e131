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


def _reference_rank(rank: int, world: int, port: int, out):
    import contextlib
    import io

    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--gpus", str(world), "--steps", "1", "--warmup", "3"])
    out[rank] = buf.getvalue()


def test_reference_arm_prints_once_under_two_ranks():
    """The reference arm (the oracle on host cores) runs on rank 0 only and
    prints one JSON line with the contract's keys; rank 1 prints nothing."""
    import json

    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_reference_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[1] == ""
    lines = out[0].strip().splitlines()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "rows/s" and d["value"] > 0
    assert d["n_gpus"] == world and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
