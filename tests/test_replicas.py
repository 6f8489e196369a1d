"""The multi-GPU face of bench.py: every rank times its own share of the rows (world copies of
the workload, sharded), the step time is the slowest rank's and the bytes are every rank's own,
summed.  The cross-rank arithmetic on two gloo ranks on the CPU, and the shares themselves."""
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
        ms_step = 2.0 if rank == 0 else 3.0  # rank 1 is the slower one
        ms_max, value = bench.combine_ranks(ms_step, 6_000_000 if rank == 0 else 6_000_000, dist, torch.device("cpu"))
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


@pytest.mark.parametrize("name", ["indexer_bf16_4096x2048_causal_k512_gather", "sampling_f32_256x131072_k4096_nan",
                                  "indexer_bf16_3x4096x16384_levels64_k2048_gather"])
@pytest.mark.parametrize("world", [1, 2, 4])
def test_shares_cover_every_copy_once(name, world):
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import synthetic as syn
    w = syn.workload(name, rows=None)
    R = w["rows"]
    seen = []
    for rank in range(world):
        grows, pieces, mode = bench.shard_plan(w, rank, world)
        assert mode == ("dual_chunk" if w["row_end"] is not None else "blocks")
        assert pieces[0][0] == 0 and pieces[-1][1] == len(grows)
        assert all(pieces[i][1] == pieces[i + 1][0] for i in range(len(pieces) - 1))
        if w.get("key") is not None:
            rpb = w["rows_per_batch"]
            for lo, hi, b0, b1 in pieces:  # a call's rows lie in its key batches
                g0, g1 = grows[lo], grows[hi - 1]
                assert b0 * rpb <= g0 and g1 < b1 * rpb and (g1 - g0 + 1) == hi - lo
        seen.append(grows)
    allrows = np.sort(np.concatenate(seen))
    assert (allrows == np.arange(R * world)).all()
    if world == 1:
        assert len(pieces) == 1  # one GPU: the whole workload in one call
