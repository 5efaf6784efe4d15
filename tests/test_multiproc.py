"""The N > 1 benchmark path on CPU: two gloo ranks, each an independent
replica of the layer (the layer has no exchange step, so the ranks share
nothing but the timing reduction).  Rank 0 must report the whole-job rate
from the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = [120.0, 200.0][rank]
    mx = bench.reduce_max_ms(my_ms)
    val = bench.aggregate_gbs(world, 1_000_000, 10, mx)
    dist.barrier()
    q.put((rank, mx, val))
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, val in res:
        assert mx == 200.0
        assert val == pytest.approx(2 * 1_000_000 * 10 / 0.2 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_ms(3.5) == 3.5
    assert bench.aggregate_gbs(1, 2e9, 1, 1000.0) == pytest.approx(2.0)
