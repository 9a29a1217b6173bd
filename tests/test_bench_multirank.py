"""The multi-rank path of bench.py (replicas, one per GPU) on CPU ranks with
gloo: every rank reports its own elapsed time, the job time is the maximum,
and the value counts the tokens of all ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, rank, world)
    elapsed = [10.0, 25.0, 17.5][rank]
    value, t = bench.aggregate(world, 8192, 4, elapsed, dist, "cpu")
    dist.barrier()
    q.put((rank, value, t))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_replica_aggregation_takes_max_over_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    tmax = max([10.0, 25.0, 17.5][:world])
    for rank, value, t in res:
        assert t == tmax
        assert value == pytest.approx(world * 8192 * 4 / (tmax / 1e3))


def test_single_rank_aggregation_is_local():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    v, t = bench.aggregate(1, 100, 10, 2.0)
    assert t == 2.0 and v == pytest.approx(100 * 10 / 2e-3)
