"""The N > 1 host path of bench.py with two gloo ranks on CPU (no GPU).

Rows are independent, so ranks shard the batch with no data-path collective;
the only exchange is the max-over-ranks timing reduction.
"""

import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    secs = bench.max_over_ranks(1.0 + rank, dist, "cpu")
    w = bench.rank_workload(8, "paged", rank)
    out = oracle.run(w, threads=1)
    q.put((rank, secs, w.scores[0, :4].tolist(), out.shape))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows_and_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]          # every rank sees the max
    assert res[0][2] != res[1][2]                     # each rank has its own rows
    assert all(r[3] == (8, 1024) for r in res)
