"""Row sharding over several GPUs (gather_radix_select_gb300.shard).

The partition, the cut at batch boundaries and the assembly are host logic;
they are checked here on the CPU, and end to end on two gloo ranks that each
compute their own pieces with the oracle (a stand-in for the library call
here only: the product module never imports the oracle) and assemble
everyone's pieces.  The CUDA path through the same sharded entry runs in the
gpu-marked test at the end.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synthetic as syn
from gather_radix_select_gb300 import shard

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("rows", [0, 1, 5, 8, 4096, 12289])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("mode", ["blocks", "dual_chunk"])
def test_partition_covers_every_row_once(rows, world, mode):
    parts = shard.partition_rows(rows, world, mode)
    assert len(parts) == world
    got = np.concatenate([shard.rows_of(r) for r in parts]) if rows else np.zeros(0)
    assert sorted(got.tolist()) == list(range(rows))
    sizes = [len(shard.rows_of(r)) for r in parts]
    assert max(sizes) - min(sizes) <= (1 if mode == "blocks" else 2)
    for r in parts:  # each rank's ranges are in row order and disjoint
        assert all(r[i][1] <= r[i + 1][0] for i in range(len(r) - 1))


def test_dual_chunk_evens_out_causal_rows():
    # causal row ends of the indexer workload: n_i = min(2048, i // 2 + 1); work ~ n_i
    rows = 4096
    n = np.minimum(2048, np.arange(rows) // 2 + 1)
    for world in (2, 4, 8):
        def spread(mode):
            w = [n[shard.rows_of(r)].sum() for r in shard.partition_rows(rows, world, mode)]
            return max(w) / (sum(w) / world)
        assert spread("dual_chunk") < 1.02
        assert spread("blocks") > 1.1   # the last block holds the longest rows
    # pure causal rows (n_i = i + 1): dual chunk is balanced up to the chunk rounding
    n = np.arange(1, 8193)
    w = [n[shard.rows_of(r)].sum() for r in shard.partition_rows(8192, 4, "dual_chunk")]
    assert max(w) / min(w) < 1.001


def test_split_at_batches():
    pieces = shard.split_at_batches([(3, 17), (20, 21), (31, 40)], 8)
    assert pieces == [(3, 8, 0), (8, 16, 1), (16, 17, 2), (20, 21, 2), (31, 32, 3), (32, 40, 4)]
    for s, e, b in pieces:
        assert b * 8 <= s < e <= (b + 1) * 8
    with pytest.raises(ValueError):
        shard.split_at_batches([(0, 4)], 0)
    # whole batches go to one call; parts of a batch to their own
    assert shard.call_pieces([(0, 24), (26, 40)], 8) == [(0, 24, 0, 3), (26, 32, 3, 4), (32, 40, 4, 5)]
    assert shard.call_pieces([(4, 20)], 8) == [(4, 8, 0, 1), (8, 16, 1, 2), (16, 20, 2, 3)]
    assert shard.partition_rows(10, 1, "dual_chunk") == [[(0, 10)]]
    assert shard.partition_rows(9, 3, "dual_chunk")[1] == [(1, 3), (6, 7)]  # chunks 1 and 4 of [0,1,3,4,6,7,9]


def test_assemble_puts_pieces_in_row_order_and_finds_gaps():
    rows, k = 10, 3
    full = np.arange(rows * k).reshape(rows, k)
    ps = [shard.Piece(s, e, None, full[s:e], None) for s, e in [(6, 10), (0, 2), (2, 6)]]
    _, idx, _ = shard.assemble(ps, rows, np.concatenate)
    assert (idx == full).all()
    with pytest.raises(ValueError):
        shard.assemble(ps[:2], rows, np.concatenate)  # a gap
    with pytest.raises(ValueError):
        shard.assemble(ps + [shard.Piece(5, 7, None, full[5:7], None)], rows, np.concatenate)  # an overlap


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    # causal bf16 score rows over two batches, with a key to gather from: a small copy of the
    # indexer workload's structure
    rows, cols, k, b, d, ng = 64, 96, 8, 2, 16, 5
    x = syn.normal_rows(77, rows, cols, "bf16")
    end = np.minimum(cols, np.arange(rows) * 3 // 2 + 1).astype(np.int32)
    key = syn.normal_rows(78, b * cols, d, "bf16").reshape(b, cols, d)
    return x, end, key, rows, cols, k, b, d, ng


def _oracle_compute(x, end, key, k, ng):
    import oracle

    def compute(s, e, batches):
        b0, b1 = batches
        idx, bits, _ = oracle.topk(x[s:e], "bf16", k, row_end=end[s:e], sorted_index=True)
        gth, _ = oracle.gather_rows(np.ascontiguousarray(key[b0:b1]), idx[:, :ng], b1 - b0)
        return bits, idx, gth
    return compute


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from gather_radix_select_gb300 import shard as sh
        x, end, key, rows, cols, k, b, d, ng = _case()
        ranges = sh.partition_rows(rows, world, "dual_chunk")[rank]
        mine = sh.run_rank(_oracle_compute(x, end, key, k, ng), ranges, rows_per_batch=rows // b)
        everyone = [None] * world
        dist.all_gather_object(everyone, mine)
        vals, idx, gth = sh.assemble([p for ps in everyone for p in ps], rows, np.concatenate)
        q.put((rank, vals, idx, gth))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_assemble_the_whole_answer():
    import oracle
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    x, end, key, rows, cols, k, b, d, ng = _case()
    want_idx, want_bits, _ = oracle.topk(x, "bf16", k, row_end=end, sorted_index=True)
    want_g, _ = oracle.gather_rows(key, want_idx[:, :ng], b)
    for _, vals, idx, gth in got:
        assert (idx == want_idx).all() and (vals == want_bits).all() and (gth == want_g).all()


@pytest.mark.gpu
@pytest.mark.parametrize("world", [1, 2, 3])
def test_library_through_the_sharded_entry(world):
    # the CUDA path, rank by rank on one GPU (no collective is involved: each rank's pieces are
    # independent calls), assembled, equals the plain fused call
    import gather_radix_select_gb300 as g
    rows, cols, k, b, d, ng = 768, 4096, 256, 3, 128, 64
    xb = syn.normal_rows(91, rows, cols, "bf16")
    end = np.minimum(cols, np.arange(rows) * 7 + 1).astype(np.int32) % (cols + 1)
    kb = syn.normal_rows(92, b * cols, d, "bf16").reshape(b, cols, d)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    e = torch.from_numpy(end).cuda()
    key = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda()
    v0, i0, g0 = g.topk_gather(x, k, key, ng, end=e, sorted_index=True, return_value=True)
    pieces = []
    compute = shard.topk_pieces(x, k, end=e, key=key, n_gather=ng, sorted_index=True, return_value=True)
    for r in shard.partition_rows(rows, world, "dual_chunk"):
        pieces += shard.run_rank(compute, r, rows_per_batch=rows // b)
    v1, i1, g1 = shard.assemble(pieces, rows, torch.cat)
    torch.cuda.synchronize()
    assert torch.equal(i0.cpu(), i1.cpu())
    assert torch.equal(v0.cpu().view(torch.int16), v1.cpu().view(torch.int16))
    assert torch.equal(g0.cpu().view(torch.int16), g1.cpu().view(torch.int16))
