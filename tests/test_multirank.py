"""The benchmark's multi-rank logic (replicas, weak scaling) on CPU with gloo, world size 2.

Each rank runs its own replica; the only cross-rank traffic is the timing
barrier and the max / sum of per-rank numbers.  The reference arm runs on
rank 0 only; other ranks exit 0 without output.
"""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (world, rank, rank)
        bench.barrier(world)
        mx = bench.max_over_ranks(10.0 + rank, world, "cpu")
        sm = bench.sum_over_ranks(100.0 * (rank + 1), world, "cpu")

        class Args:
            gpus = world
            steps = 1
            warmup = 3

        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.run_reference(Args) if rank != 0 else 0
        results[rank] = (mx, sm, rc, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_rank_replica_aggregation():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        results = manager.dict()
        mp.start_processes(_worker, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
        res = dict(results)
    assert res[0][0] == res[1][0] == 11.0
    assert res[0][1] == res[1][1] == 300.0
    # the reference arm on a non-zero rank does nothing and exits 0
    assert res[1][2] == 0 and res[1][3] == ""
