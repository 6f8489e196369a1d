"""Block-level candidate selection with its gather (sel_block_topk_gather) against the
oracle: positions element by element, gathered key rows bitwise."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import to_bits, to_torch

pytestmark = pytest.mark.gpu


def run(scores_bits, dtype, topk_blocks, block_size, pos_end=None, key_bits=None):
    import gather_radix_select_gb300 as g
    scores = to_torch(scores_bits, dtype)
    pe = None if pos_end is None else torch.from_numpy(pos_end).cuda()
    key = None if key_bits is None else to_torch(key_bits, "bf16")
    nan = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos, out = g.block_topk_gather(scores, topk_blocks, block_size, pos_end=pe, key=key, nan_flag=nan,
                                   err_flag=err)
    torch.cuda.synchronize()
    return pos.cpu().numpy().astype(np.int64), out, int(nan.item()), int(err.item())


CASES = [
    # (dtype, rows, n_blocks, topk_blocks, block_size)
    ("bf16", 40, 32, 16, 64),
    ("f32", 33, 7, 3, 5),
    ("bf16", 17, 300, 100, 3),
    ("f32", 9, 5000, 64, 2),
    ("bf16", 5, 16, 40, 8),       # more blocks wanted than exist
    ("f32", 6, 1, 1, 128),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_block_candidates_match_oracle(case):
    dtype, rows, n_blocks, tb, bs = case
    rng = np.random.default_rng(rows * 7 + n_blocks)
    v = rng.standard_normal((rows, n_blocks)).astype(np.float32)
    v[::3] = np.round(v[::3] * 2) / 2  # ties on some rows
    e = syn.elem_bytes(dtype)
    stride = (n_blocks * e + 15) // 16 * 16 // e
    bits = np.zeros((rows, stride), dtype=np.uint32 if dtype == "f32" else np.uint16)
    bits[:, :n_blocks] = syn.f32_to_bits(v) if dtype == "f32" else syn.f32_to_bf16_bits(v)
    pe = rng.integers(-3, n_blocks * bs + 5, size=rows).astype(np.int32)
    pe[0], pe[-1] = n_blocks * bs, 0
    comp_len = n_blocks * bs
    key = syn.f32_to_bf16_bits(rng.standard_normal((1, comp_len, 64)).astype(np.float32))
    import gather_radix_select_gb300 as g
    scores = to_torch(bits, dtype)[:, :n_blocks]
    pos, out = g.block_topk_gather(scores, tb, bs, pos_end=torch.from_numpy(pe).cuda(), key=to_torch(key, "bf16"))
    torch.cuda.synchronize()
    want, nan = oracle.block_candidates(np.ascontiguousarray(bits[:, :n_blocks]), dtype, tb, bs, pos_end=pe)
    assert not nan.any()
    assert (pos.cpu().numpy().astype(np.int64) == want).all()
    gw, bad = oracle.gather_rows(key, want, 1)
    assert bad == 0
    assert (to_bits(out) == gw).all()


def test_block_candidates_positions_only_and_no_end():
    rng = np.random.default_rng(3)
    bits = syn.f32_to_bf16_bits(rng.standard_normal((8, 64)).astype(np.float32))
    pos, out, nan, err = run(bits, "bf16", 5, 16)
    assert out is None and nan == 0 and err == 0
    want, _ = oracle.block_candidates(bits, "bf16", 5, 16)
    assert (pos == want).all()


def test_block_candidates_workload():
    # 1024 query rows, 32 blocks of 64 over compressed length 2048, 16 blocks -> 1024 positions a
    # row, causal ends, gather of the 128-wide key rows
    w = syn.block_candidates_workload()
    pos, out, nan, err = run(w["scores"], "bf16", w["topk_blocks"], w["block_size"], w["pos_end"], w["key"])
    assert nan == 0 and err == 0
    want, _ = oracle.block_candidates(w["scores"], "bf16", w["topk_blocks"], w["block_size"], w["pos_end"])
    assert (pos == want).all()
    rows = np.linspace(0, w["rows"] - 1, 24).astype(np.int64)
    gw, _ = oracle.gather_rows(w["key"], want[rows], 1)
    assert (to_bits(out[torch.from_numpy(rows).cuda()]) == gw).all()
    # every row, on the device: the gathered rows are the key rows at the safe positions
    flat = torch.from_numpy(pos).cuda().clamp(min=0).reshape(-1)
    key = to_torch(w["key"], "bf16")[0]
    assert torch.equal(out.view(torch.int16), torch.index_select(key, 0, flat).view(torch.int16).view(out.shape))


def test_block_candidates_nan_row_flagged():
    v = np.random.default_rng(4).standard_normal((3, 40)).astype(np.float32)
    v[1, 7] = np.nan
    bits = syn.f32_to_bits(v)
    pos, _, nan, err = run(bits, "f32", 8, 4)
    assert nan == 1 and err == 0
    want, o_nan = oracle.block_candidates(bits, "f32", 8, 4)
    assert o_nan.tolist() == [0, 1, 0]
    assert (pos[[0, 2]] == want[[0, 2]]).all()
    # the flagged row still lists in-range positions then -1
    p = pos[1]
    m = int((p >= 0).sum())
    assert (p[:m] >= 0).all() and (p[m:] == -1).all() and (p[:m] < 160).all()
