"""The N>1 path of bench.py: independent replicas, max time over ranks, units summed (gloo, 2 ranks, CPU)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [0.5, 0.8][rank]
    units = [100.0, 300.0][rank]
    t, u = bench.reduce_replicas(elapsed, units, world)
    bench.barrier(world)
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_reduce_replicas_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u in got:
        assert t == pytest.approx(0.8)     # slowest replica
        assert u == pytest.approx(400.0)   # whole-job units


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_replicas(1.5, 7.0, 1) == (1.5, 7.0)
