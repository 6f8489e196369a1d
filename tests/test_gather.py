"""GPU parity of sel_gather_rows and sel_topk_gather (through the C ABI).

The gather list follows the unit tests named by the MindSpore hyper-parallel
pull request "perf/gather-index-select": equality with two-tensor advanced
indexing at batch 1 and batch > 1, batches do not mix, shape and dtype, a
non-contiguous key, repeated positions -- plus -1 (safe) positions,
out-of-range positions, int32/int64 positions and the full-size workloads.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import IDX_DTYPE, check_definition_on_device, compare_with_oracle, to_bits, to_torch

pytestmark = pytest.mark.gpu


def gsel():
    import gather_radix_select_gb300 as g
    return g


def key_tensor(bits):
    return to_torch(bits, "bf16")


@pytest.mark.parametrize("b", [1, 3])
@pytest.mark.parametrize("idx_dtype", ["i32", "i64"])
def test_gather_matches_oracle(b, idx_dtype):
    comp_len, d, rows_per_b, n = 300, 128, 7, 50
    key = syn.f32_to_bf16_bits(np.random.default_rng(b).standard_normal((b, comp_len, d)).astype(np.float32))
    key = key.reshape(b, comp_len, d)
    pos = syn.gather_positions(40 + b, b * rows_per_b, n, comp_len, neg_frac=0.1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gsel().gather_rows(key_tensor(key), torch.from_numpy(pos).to(IDX_DTYPE[idx_dtype]).cuda(), err_flag=err)
    torch.cuda.synchronize()
    want, bad = oracle.gather_rows(key, pos, b)
    assert bad == 0 and int(err.item()) == 0
    assert out.shape == (b * rows_per_b, n, d) and out.dtype == torch.bfloat16
    assert (to_bits(out) == want).all()
    # the flat form: one index_select over the batch-flattened key
    flat = key_tensor(key).reshape(b * comp_len, d)
    fpos = (torch.arange(b * rows_per_b)[:, None] // rows_per_b) * comp_len + torch.from_numpy(pos).clamp(min=0)
    ref = torch.index_select(flat, 0, fpos.reshape(-1).cuda()).reshape(b * rows_per_b, n, d)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_batches_do_not_mix():
    b, comp_len, d = 3, 64, 64
    key = np.zeros((b, comp_len, d), dtype=np.uint16)
    for bb in range(b):
        key[bb] = syn.f32_to_bf16_bits(np.full((comp_len, d), bb + 1, np.float32))
    pos = np.tile(np.arange(comp_len, dtype=np.int32), (b * 4, 1))
    out = to_bits(gsel().gather_rows(key_tensor(key), torch.from_numpy(pos).cuda()))
    for r in range(b * 4):
        assert (out[r] == key[r // 4, 0, 0]).all()


def test_noncontiguous_key_and_repeats():
    rng = np.random.default_rng(8)
    base = syn.f32_to_bf16_bits(rng.standard_normal((2, 100, 96)).astype(np.float32)).reshape(2, 100, 96)
    kt = key_tensor(base)[:, :, 16:80]  # row stride 96, d = 64
    assert not kt.is_contiguous()
    pos = np.array([[5, 5, 5, -1, 99, 0]] * 4, dtype=np.int64)
    out = to_bits(gsel().gather_rows(kt, torch.from_numpy(pos).cuda()))
    want, _ = oracle.gather_rows(base[:, :, 16:80], pos, 2)
    assert (out == want).all()
    assert (out[0, 0] == out[0, 1]).all() and (out[0, 3] == base[0, 0, 16:80]).all()


def test_out_of_range_position_zero_row_and_flag():
    key = syn.f32_to_bf16_bits(np.ones((1, 10, 16), np.float32)).reshape(1, 10, 16)
    pos = np.array([[1, 10, 2]], dtype=np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = to_bits(gsel().gather_rows(key_tensor(key), torch.from_numpy(pos).cuda(), err_flag=err))
    assert int(err.item()) == 1
    assert (out[0, 1] == 0).all() and (out[0, 0] == key[0, 1]).all() and (out[0, 2] == key[0, 2]).all()


def test_gather_alignment_rejected():
    g = gsel()
    key = torch.zeros((1, 10, 12), dtype=torch.bfloat16, device="cuda")  # 24-byte rows
    with pytest.raises(g.SelError) as e:
        g.gather_rows(key, torch.zeros((1, 3), dtype=torch.int32, device="cuda"))
    assert e.value.status == 2


GATHER_WORKLOADS = ["indexer_bf16_4096x2048_causal_k512_gather", "indexer_bf16_3x4096x16384_levels64_k2048_gather"]


@pytest.mark.parametrize("name", GATHER_WORKLOADS)
def test_workload_gather_and_fused(name):
    g = gsel()
    w = syn.workload(name)
    x = to_torch(w["x"], w["dtype"])
    end = torch.from_numpy(w["row_end"]).cuda()
    key = key_tensor(w["key"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, idx = g.topk(x, w["k"], end=end, sorted_index=False, return_value=False)
    # separate gather of the first n_gather selected positions
    sel = idx[:, :w["n_gather"]]
    out = g.gather_rows(key, sel, err_flag=err)
    # fused selection + gather
    _, fidx, fout = g.topk_gather(x, w["k"], key, w["n_gather"], end=end, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(fidx, idx)
    assert torch.equal(fout.view(torch.int16), out.view(torch.int16))
    # the selection itself is right on every row
    nv = torch.from_numpy(np.clip(w["row_end"], 0, w["cols"]).astype(np.int64)).cuda()
    check_definition_on_device(x, nv, w["k"], idx, None, False)
    # the gather equals the oracle on sampled rows of every batch, and torch.index_select on all rows
    sel_np = sel.cpu().numpy()
    rpb = w["rows_per_batch"]
    for bb in range(w["b"]):
        rr = np.unique(np.linspace(bb * rpb, bb * rpb + rpb - 1, 8).astype(np.int64))
        want, bad = oracle.gather_rows(np.ascontiguousarray(w["key"][bb:bb + 1]), sel_np[rr], 1)
        assert bad == 0 and (to_bits(out[torch.from_numpy(rr).cuda()]) == want).all()
    flat = key.reshape(-1, w["d"])
    batch = torch.arange(w["rows"], device="cuda")[:, None] // w["rows_per_batch"]
    fpos = batch * w["comp_len"] + sel.to(torch.int64).clamp(min=0)
    ref = torch.index_select(flat, 0, fpos.reshape(-1)).reshape(out.shape)
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))
    # top-k parity with the oracle on sampled rows
    rows = np.unique(np.linspace(0, w["rows"] - 1, 24).astype(np.int64))
    compare_with_oracle(w, rows, idx.cpu().numpy()[rows], None, False)


def test_fused_small_cases_match_separate():
    g = gsel()
    rng = np.random.default_rng(12)
    for dtype, rows, cols, k, ng, b in (("bf16", 6, 3000, 100, 100, 2), ("f32", 4, 70000, 300, 64, 1),
                                        ("bf16", 9, 500, 600, 300, 3)):
        v = rng.standard_normal((rows, cols)).astype(np.float32)
        bits = syn.f32_to_bits(v) if dtype == "f32" else syn.f32_to_bf16_bits(v)
        e = syn.elem_bytes(dtype)
        stride = (cols * e + 15) // 16 * 16 // e
        padded = np.zeros((rows, stride), dtype=bits.dtype)
        padded[:, :cols] = bits
        x = to_torch(padded, dtype)[:, :cols]  # row stride padded to 16 bytes
        end = torch.from_numpy(rng.integers(0, cols + 1, size=rows).astype(np.int32)).cuda()
        key = key_tensor(syn.f32_to_bf16_bits(rng.standard_normal((b, cols, 64)).astype(np.float32)))
        vals, idx = g.topk(x, k, end=end, sorted_index=True, return_value=True)
        fvals, fidx, fout = g.topk_gather(x, k, key, ng, end=end, sorted_index=True, return_value=True)
        out = g.gather_rows(key, idx[:, :ng])
        torch.cuda.synchronize()
        assert torch.equal(fidx, idx) and torch.equal(fvals.view(torch.int16) if dtype == "bf16" else
                                                      fvals.view(torch.int32),
                                                      vals.view(torch.int16) if dtype == "bf16" else
                                                      vals.view(torch.int32))
        assert torch.equal(fout.view(torch.int16), out.view(torch.int16))


# --------------------------------------------------------------------------
# two keys at the same positions (the Indexer KL loss's index key + attention key)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("b", [1, 3])
@pytest.mark.parametrize("idx_dtype", ["i32", "i64"])
def test_gather_pair_matches_oracle(b, idx_dtype):
    comp_len, d, d2, rows_per_b, n = 300, 64, 256, 5, 70
    g = np.random.default_rng(30 + b)
    key = syn.f32_to_bf16_bits(g.standard_normal((b, comp_len, d)).astype(np.float32))
    base2 = syn.f32_to_bf16_bits(g.standard_normal((b, comp_len, d2 + 64)).astype(np.float32))
    k2 = key_tensor(base2)[:, :, 32:32 + d2]  # row stride d2 + 64: a non-contiguous second key
    assert not k2.is_contiguous()
    pos = syn.gather_positions(50 + b, b * rows_per_b, n, comp_len, neg_frac=0.1)
    pos[0, :3] = pos[0, 3]  # repeated positions
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, out2 = gsel().gather_rows_pair(key_tensor(key), k2, torch.from_numpy(pos).to(IDX_DTYPE[idx_dtype]).cuda(),
                                        err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert out.shape == (b * rows_per_b, n, d) and out2.shape == (b * rows_per_b, n, d2)
    want, bad = oracle.gather_rows(key, pos, b)
    want2, bad2 = oracle.gather_rows(base2[:, :, 32:32 + d2], pos, b)
    assert bad == 0 and bad2 == 0
    assert (to_bits(out) == want).all()
    assert (to_bits(out2) == want2).all()


def test_gather_pair_out_of_range_zero_rows_and_flag():
    key = syn.f32_to_bf16_bits(np.ones((1, 10, 16), np.float32))
    key2 = syn.f32_to_bf16_bits(np.full((1, 10, 32), 2.0, np.float32))
    pos = np.array([[1, 10, -1]], dtype=np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, out2 = gsel().gather_rows_pair(key_tensor(key), key_tensor(key2), torch.from_numpy(pos).cuda(), err_flag=err)
    out, out2 = to_bits(out), to_bits(out2)
    assert int(err.item()) == 1
    assert (out[0, 1] == 0).all() and (out2[0, 1] == 0).all()
    assert (out[0, 2] == key[0, 0]).all() and (out2[0, 2] == key2[0, 0]).all()


def test_gather_pair_full_size():
    # 1024 rows x 512 positions, index key d=128 and attention key d=512 at compressed length 2048
    w = syn.kl_pair_gather()
    key, key2 = key_tensor(w["key"]), key_tensor(w["key2"])
    pos = torch.from_numpy(w["pos"]).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, out2 = gsel().gather_rows_pair(key, key2, pos, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # every row: the flat index_select form on the device
    flat = pos.to(torch.int64).clamp(min=0).reshape(-1)
    assert torch.equal(out.view(torch.int16), torch.index_select(key[0], 0, flat).view(torch.int16).view(out.shape))
    assert torch.equal(out2.view(torch.int16),
                       torch.index_select(key2[0], 0, flat).view(torch.int16).view(out2.shape))
    # sampled rows: the oracle
    rows = np.linspace(0, w["rows"] - 1, 16).astype(np.int64)
    want, _ = oracle.gather_rows(w["key"], w["pos"][rows], 1)
    want2, _ = oracle.gather_rows(w["key2"], w["pos"][rows], 1)
    assert (to_bits(out[torch.from_numpy(rows).cuda()]) == want).all()
    assert (to_bits(out2[torch.from_numpy(rows).cuda()]) == want2).all()


@pytest.mark.parametrize("d", [48, 2560])
def test_gather_general_row_widths(d):
    # 6 and 320 16-byte vectors a row: not a power of two / wider than the CTA (the general loop)
    rng = np.random.default_rng(d)
    b, comp_len, rows_per_b, n = 2, 90, 3, 37
    key = syn.f32_to_bf16_bits(rng.standard_normal((b, comp_len, d)).astype(np.float32)).reshape(b, comp_len, d)
    key2 = syn.f32_to_bf16_bits(rng.standard_normal((b, comp_len, 16)).astype(np.float32)).reshape(b, comp_len, 16)
    pos = syn.gather_positions(7, b * rows_per_b, n, comp_len, neg_frac=0.1)
    pos[1, 3] = comp_len + 2  # out of range: zero row and error flag
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gsel().gather_rows(key_tensor(key), torch.from_numpy(pos).cuda(), err_flag=err)
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    p1, p2 = gsel().gather_rows_pair(key_tensor(key), key_tensor(key2), torch.from_numpy(pos).cuda(), err_flag=err2)
    torch.cuda.synchronize()
    want, bad = oracle.gather_rows(key, pos, b)
    want2, _ = oracle.gather_rows(key2, pos, b)
    assert bad == 1 and int(err.item()) == 1 and int(err2.item()) == 1
    assert (to_bits(out) == want).all()
    assert (to_bits(p1) == want).all() and (to_bits(p2) == want2).all()
