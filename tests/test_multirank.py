"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Rows are independent, so N GPUs run N independent batches (weak scaling, no
data-path collective); the only cross-rank steps are the barrier around the
timed region and the reductions that turn per-rank times and row counts into
the job's number: the slowest rank's time and the sum of all ranks' rows.
"""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier()
        t = bench.max_over_ranks(0.5 + rank, None)  # rank 1 is the slowest
        rows = bench.sum_over_ranks(128.0, None)
        out.put((rank, t, rows))
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, rows in res:
        assert t == pytest.approx(1.5) and rows == pytest.approx(256.0)


def test_single_rank_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.25) == 3.25 and bench.sum_over_ranks(7.0) == 7.0
    assert bench.dist_env()[0] in (1, int(os.environ.get("WORLD_SIZE", "1")))
