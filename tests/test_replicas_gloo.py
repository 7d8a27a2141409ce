"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank runs
an independent replica; the job's time is the maximum over ranks and its work
the sum, with no data exchanged between replicas."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        elapsed = [1.5, 2.25][rank]
        units = [100.0, 40.0][rank]
        t, u = bench.reduce_over_ranks(elapsed, units)
        bench.barrier()
        q.put((rank, t, u))
    finally:
        dist.destroy_process_group()


def test_replica_time_is_max_and_work_is_sum():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, u in got:
        assert t == pytest.approx(2.25)
        assert u == pytest.approx(140.0)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.0, 7.0) == (3.0, 7.0)
