"""The multi-rank path of bench.py on the CPU: world size 2 over gloo.

Each rank verifies its own requests (no collective on the data path); the
only cross-rank steps are a barrier and the max of the per-step time, and
the reported throughput is all ranks' rows over the slowest rank's time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    ms = [0.120, 0.135][rank]               # this rank's time per step
    dist.barrier()
    ms_max = bench.reduce_max(ms, world, "cpu")
    value = bench.aggregate(ms_max, 64 * 16, world)
    q.put((rank, ms_max, value))
    dist.destroy_process_group()


def test_two_ranks_max_time_and_weak_scaling_sum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value in out:
        assert ms_max == pytest.approx(0.135)
        assert value == pytest.approx(2 * 64 * 16 / 0.135e-3)


def test_single_rank_aggregate():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.5, 1, "cpu") == 1.5
    assert bench.aggregate(0.1, 1024, 1) == pytest.approx(1024 / 1e-4)
