"""The multi-rank bench logic on CPU: two gloo ranks, the whole-job time is
the slowest rank's and the value aggregates every rank's bytes."""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, str(ROOT))
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + rank, 30.0 - rank, 1.5 * (rank + 1)]
    got = bench.max_over_ranks(mine)
    value = bench.whole_job_gbs(world, 1_000_000_000, got[0])
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, value))


def test_two_rank_aggregation():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q))
             for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in results:
        assert got == [11.0, 30.0, 3.0]
        # 2 ranks x 1 GB in 11 ms
        assert value == pytest.approx(2 * 1e9 / 11e-3 / 1e9)


def test_single_process_is_identity():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks([1.0, 2.0]) == [1.0, 2.0]
