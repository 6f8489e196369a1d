"""The multi-GPU face of bench.py is replicas: every rank runs the same workload and the
step time is the slowest rank's.  Its cross-rank arithmetic, on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_step = 2.0 if rank == 0 else 3.0  # rank 1 is the slower replica
        ms_max, value = bench.combine_ranks(ms_step, 6_000_000, dist, torch.device("cpu"))
        q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms_max, value in got:
        assert ms_max == pytest.approx(3.0)
        # 2 ranks x 6 MB in 3 ms = 4 GB/s
        assert value == pytest.approx(4.0)


def test_single_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ms_max, value = bench.combine_ranks(1.5, 3_000_000, None, torch.device("cpu"))
    assert ms_max == 1.5 and value == pytest.approx(2.0)
