"""Pins for the CPU oracle (no GPU).

The oracle (``oracle/ref.c``) is held to things other than itself:

* the rank definition of top-k, evaluated by O(n^2) brute force on tiny rows;
* hand-worked closed forms (ties, -0/+0, short rows, fills);
* library routines for the special cases they cover (numpy argmax for k=1,
  numpy argpartition / torch.topk on tie-free rows, numpy advanced indexing
  and torch index_select for the gather);
* the example shapes printed by the DeepSelect tutorial (tests/golden);
* mutation checks: a copy of ref.c with a planted mistake must fail a pin.
"""
import json
import os
import subprocess
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32bits(vals):
    return np.asarray(vals, dtype=np.float32).view(np.uint32)


def bf16bits(vals):
    return syn.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def tiny_row(kind, n, rng, dtype):
    if kind == "normal":
        v = rng.standard_normal(n).astype(np.float32)
    elif kind == "equal":
        v = np.full(n, 1.5, dtype=np.float32)
    elif kind == "two_level":
        v = np.where(rng.random(n) < 0.5, 1.0, -2.0).astype(np.float32)
    elif kind == "zeros":
        v = np.where(rng.random(n) < 0.5, 0.0, -0.0).astype(np.float32)
    elif kind == "inf":
        v = rng.choice(np.array([np.inf, -np.inf, 0.0, -0.0, 1.0, -1.0], dtype=np.float32), size=n)
    elif kind == "small_ints":
        v = rng.integers(-3, 4, size=n).astype(np.float32)
    else:
        raise ValueError(kind)
    return f32bits(v) if dtype == "f32" else bf16bits(v)


KINDS = ("normal", "equal", "two_level", "zeros", "inf", "small_ints")


def selected_sorted(idx_row, valid_count):
    head = [int(i) for i in idx_row[:valid_count]]
    return sorted(head)


# --------------------------------------------------------------------------
# brute force on tiny rows, every k
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", KINDS)
def test_oracle_matches_rank_brute_force(dtype, kind):
    rng = np.random.default_rng(7 + KINDS.index(kind) + (100 if dtype == "bf16" else 0))
    for n in (0, 1, 2, 3, 5, 8, 13, 31, 32, 33, 64):
        cols = max(n, 1)
        x = np.zeros((1, cols), dtype=np.uint32 if dtype == "f32" else np.uint16)
        if n:
            x[0, :n] = tiny_row(kind, n, rng, dtype)
        vals = oracle.bits_to_values(x[0], dtype)
        for k in range(1, 71):
            for row_end in (None, n, n // 2):
                re_arr = None if row_end is None else np.array([row_end], dtype=np.int32)
                idx, bits, nan = oracle.topk(x, dtype, k, row_end=re_arr, sorted_index=True, cols=n)
                nn = n if row_end is None else row_end
                want = oracle.brute_topk_row(vals, nn, k)
                got = [int(i) for i in idx[0] if i >= 0]
                assert got == want, (kind, n, k, row_end)
                # fills at the tail, exactly k - len(want) of them
                assert all(int(i) == -1 for i in idx[0][len(want):])
                assert (bits[0][:len(want)] == x[0][want]).all()
                assert nan[0] == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_oracle_unsorted_order_is_value_descending(dtype):
    rng = np.random.default_rng(11)
    x = tiny_row("small_ints", 40, rng, dtype)[None, :]
    idx, bits, _ = oracle.topk(x, dtype, 17, sorted_index=False)
    v = oracle.bits_to_values(x[0], dtype)[idx[0]]
    assert np.all(np.diff(v) <= 0)
    # equal values are listed by ascending index
    for a, b in zip(range(16), range(1, 17)):
        if v[a] == v[b]:
            assert idx[0][a] < idx[0][b]


def stable_sort_order(v_f32, n, k):
    """Value order by a library routine: a stable descending torch.sort on CPU
    (ties keep index order, NaN ranks above every number, -0 == +0)."""
    t = torch.sort(torch.from_numpy(np.ascontiguousarray(v_f32[:n])), descending=True, stable=True)
    got = t.indices[:k].tolist()
    return got + [-1] * (k - len(got))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["small_ints", "two_level", "normal"])
def test_value_order_matches_stable_torch_sort(dtype, kind):
    rng = np.random.default_rng(23)
    rows, cols = 6, 300
    x = np.stack([tiny_row(kind, cols, rng, dtype) for _ in range(rows)])
    end = np.array([300, 299, 64, 65, 1, 0], np.int32)
    for k in (1, 7, 64, 65, 301):
        idx, bits, nan = oracle.topk(x, dtype, k, row_end=end, sorted_value=True)
        for r in range(rows):
            v = oracle.bits_to_values(x[r], dtype).astype(np.float32)
            assert idx[r].tolist() == stable_sort_order(v, int(end[r]), k), (k, r)
            n_ok = min(int(end[r]), k)
            assert (bits[r][:n_ok] == x[r][idx[r][:n_ok]]).all()
            assert (bits[r][n_ok:] == oracle.value_fill_bits(dtype)).all()
        assert not nan.any()


def test_value_order_short_row_nan_and_signed_zero():
    # short rows are not checked for NaN; in value order a NaN ranks above every number
    v = np.array([1.0, np.nan, -0.0, 0.0, 2.0, -np.nan, 2.0, -np.inf], dtype=np.float32)
    x = f32bits(v)[None, :].copy()
    idx, bits, nan = oracle.topk(x, "f32", 10, sorted_value=True)
    assert idx[0].tolist() == [1, 5, 4, 6, 0, 2, 3, 7, -1, -1]
    assert idx[0].tolist() == stable_sort_order(v, 8, 10)
    assert nan[0] == 0
    assert bits[0][5] == 0x80000000 and bits[0][6] == 0  # -0 (column 2) before +0 (column 3): a tie
    with pytest.raises(ValueError):
        oracle.topk(x, "f32", 3, sorted_index=True, sorted_value=True)


# --------------------------------------------------------------------------
# block-level candidate positions
# --------------------------------------------------------------------------

def test_block_candidates_handworked():
    # blocks of 3 positions; scores 0.5, 2.0, 1.0, 2.0; valid positions [0, 11)
    v = f32bits([0.5, 2.0, 1.0, 2.0])[None, :]
    pos, nan = oracle.block_candidates(v, "f32", 2, 3, pos_end=np.array([11], np.int32))
    # blocks 1 and 3 tie at 2.0 and beat the rest; block 3 holds 9, 10 (11 is past the end)
    assert pos[0].tolist() == [3, 4, 5, 9, 10, -1] and nan[0] == 0
    # end inside block 1: candidates are blocks 0 and 1 only
    pos, _ = oracle.block_candidates(v, "f32", 2, 3, pos_end=np.array([4], np.int32))
    assert pos[0].tolist() == [0, 1, 2, 3, -1, -1]
    # no valid position / end past the last block
    pos, _ = oracle.block_candidates(v, "f32", 1, 3, pos_end=np.array([0], np.int32))
    assert pos[0].tolist() == [-1, -1, -1]
    pos, _ = oracle.block_candidates(v, "f32", 1, 3, pos_end=np.array([99], np.int32))
    assert pos[0].tolist() == [3, 4, 5]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_block_candidates_match_brute_force(dtype):
    # chosen blocks by the O(n^2) rank definition; positions by numpy repeat / nonzero
    rng = np.random.default_rng(41)
    for trial in range(60):
        n_blocks = int(rng.integers(1, 12))
        bs = int(rng.integers(1, 6))
        tb = int(rng.integers(1, n_blocks + 3))
        kind = ["small_ints", "two_level", "normal"][trial % 3]
        x = tiny_row(kind, n_blocks, rng, dtype)[None, :]
        pe = int(rng.integers(0, n_blocks * bs + 3))
        pos, _ = oracle.block_candidates(x, dtype, tb, bs, pos_end=np.array([pe], np.int32))
        pe_c = min(pe, n_blocks * bs)
        n_cand = -(-pe_c // bs)
        chosen = np.zeros(n_blocks, bool)
        chosen[oracle.brute_topk_row(oracle.bits_to_values(x[0], dtype), n_cand, tb)] = True
        valid = np.repeat(chosen, bs) & (np.arange(n_blocks * bs) < pe_c)
        want = np.nonzero(valid)[0].tolist()
        assert pos[0].tolist() == want + [-1] * (tb * bs - len(want)), (trial, n_blocks, bs, tb, pe)


def test_block_candidates_all_blocks_is_every_valid_position():
    rng = np.random.default_rng(43)
    x = tiny_row("normal", 20, rng, "bf16")
    x = np.stack([x, x, x])
    pe = np.array([0, 37, 500], np.int32)
    pos, _ = oracle.block_candidates(x, "bf16", 20, 8, pos_end=pe)
    for r in range(3):
        n = min(int(pe[r]), 160)
        assert pos[r].tolist() == list(range(n)) + [-1] * (160 - n)


# --------------------------------------------------------------------------
# hand-worked closed forms
# --------------------------------------------------------------------------

def test_handworked_distinct_values():
    x = f32bits([3, 1, 4, 1, 5, 9, 2, 6])[None, :]
    idx, bits, _ = oracle.topk(x, "f32", 3, sorted_index=True)
    assert idx.tolist() == [[4, 5, 7]]
    assert bits.view(np.uint32).tolist() == [f32bits([5, 9, 6]).tolist()]
    idx, _, _ = oracle.topk(x, "f32", 3, sorted_index=False)
    assert idx.tolist() == [[5, 7, 4]]


def test_handworked_ties_smaller_index_wins():
    x = f32bits([2, 7, 7, 1, 7])[None, :]
    idx, _, _ = oracle.topk(x, "f32", 2, sorted_index=True)
    assert idx.tolist() == [[1, 2]]
    idx, _, _ = oracle.topk(x, "f32", 4, sorted_index=True)
    assert idx.tolist() == [[0, 1, 2, 4]]


def test_handworked_negative_and_positive_zero_tie():
    # -0 == +0 under float comparison, so the smaller index wins either way
    for vals in ([-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]):
        x = f32bits(vals)[None, :]
        idx, bits, _ = oracle.topk(x, "f32", 1)
        assert idx.tolist() == [[0]]
        assert int(bits[0, 0]) == int(f32bits(vals)[0])  # raw bits are kept (sign of zero)


def test_handworked_short_row_fills():
    # "Working with variable-length rows": a row shorter than k is filled
    x = f32bits([5, 4, 3, 2, 1])[None, :]
    idx, bits, nan = oracle.topk(x, "f32", 4, row_end=np.array([3], np.int32), sorted_index=False)
    assert idx.tolist() == [[0, 1, 2, -1]]
    assert bits[0].tolist() == f32bits([5, 4, 3]).tolist() + [0xFF800000]
    xb = bf16bits([5, 4, 3, 2, 1])[None, :]
    idx, bits, nan = oracle.topk(xb, "bf16", 6, sorted_index=True)
    assert idx.tolist() == [[0, 1, 2, 3, 4, -1]]
    assert bits[0].tolist()[-1] == 0xFF80
    assert oracle.value_fill_bits("f32") == 0xFF800000 and oracle.value_fill_bits("bf16") == 0xFF80


def test_row_end_clamped_and_zero():
    x = f32bits(np.arange(10, dtype=np.float32))[None, :].repeat(4, axis=0)
    idx, _, _ = oracle.topk(x, "f32", 3, row_end=np.array([-5, 0, 2, 99], np.int32), sorted_index=True)
    assert idx[0].tolist() == [-1, -1, -1]
    assert idx[1].tolist() == [-1, -1, -1]
    assert idx[2].tolist() == [0, 1, -1]
    assert idx[3].tolist() == [7, 8, 9]


def test_stride_padding_is_never_read():
    # columns beyond cols (row padding) hold huge values that must never be selected
    rng = np.random.default_rng(3)
    v = rng.standard_normal((3, 40)).astype(np.float32)
    v[:, 33:] = 1e30
    x = f32bits(v)
    idx, _, _ = oracle.topk(x, "f32", 5, cols=33, sorted_index=True)
    assert (idx < 33).all()
    idx2, _, _ = oracle.topk(np.ascontiguousarray(x[:, :33]), "f32", 5, sorted_index=True)
    assert (idx == idx2).all()


# --------------------------------------------------------------------------
# NaN check ("NaN handling": rows with valid length <= k are not checked)
# --------------------------------------------------------------------------

def test_nan_flag_only_on_checked_rows():
    v = np.ones((3, 8), dtype=np.float32)
    v[0, 2] = np.nan          # long row (n=8 > k=4): checked
    v[1, 7] = np.nan          # n = 4 = k: not checked
    v[2, 6] = np.nan          # NaN beyond row_end=5: outside the row
    x = f32bits(v)
    _, _, nan = oracle.topk(x, "f32", 4, row_end=np.array([8, 4, 5], np.int32))
    assert nan.tolist() == [1, 0, 0]
    xb = bf16bits(v)
    _, _, nan = oracle.topk(xb, "bf16", 4, row_end=np.array([8, 8, 5], np.int32))
    assert nan.tolist() == [1, 1, 0]


# --------------------------------------------------------------------------
# library routines for special cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_k1_is_numpy_argmax(dtype):
    rng = np.random.default_rng(5)
    for kind in KINDS:
        if kind == "zeros":
            continue  # argmax on -0/+0 compares equal too, but keep the check to real ties
        x = np.stack([tiny_row(kind, 50, rng, dtype) for _ in range(6)])
        idx, _, _ = oracle.topk(x, dtype, 1)
        vals = oracle.bits_to_values(x, dtype)
        assert idx[:, 0].tolist() == np.argmax(vals, axis=1).tolist()


def test_tie_free_rows_match_argpartition_and_torch_topk():
    rng = np.random.default_rng(9)
    v = rng.permutation(5000 * 3).astype(np.float32).reshape(3, 5000) - 7000.0
    x = f32bits(v)
    for k in (1, 7, 64, 1000, 4096):
        idx, bits, _ = oracle.topk(x, "f32", k, sorted_index=True)
        part = np.sort(np.argpartition(-v, k - 1, axis=1)[:, :k], axis=1)
        assert (idx == part).all()
        tv, ti = torch.topk(torch.from_numpy(v), k, dim=1)
        assert (idx == np.sort(ti.numpy(), axis=1)).all()
        assert (bits.view(np.uint32) == f32bits(v)[np.arange(3)[:, None], idx]).all()


def test_k_at_least_n_is_all_columns():
    rng = np.random.default_rng(1)
    x = f32bits(rng.standard_normal((2, 30)).astype(np.float32))
    for k in (30, 31, 4096):
        idx, bits, _ = oracle.topk(x, "f32", k, sorted_index=False)
        assert idx[:, :30].tolist() == [list(range(30))] * 2
        assert (idx[:, 30:] == -1).all()
        assert (bits[:, :30] == x).all()


# --------------------------------------------------------------------------
# invariants on samples of every named workload
# --------------------------------------------------------------------------

def check_invariants(w, idx, bits, nan):
    x = w["x"]
    dtype = w["dtype"]
    vals = oracle.bits_to_values(x, dtype)
    for r in range(w["rows"]):
        if nan[r]:
            continue  # selection in a row holding a NaN is unspecified
        n = w["cols"] if w["row_end"] is None else int(min(max(w["row_end"][r], 0), w["cols"]))
        k = w["k"]
        row = idx[r]
        valid = min(n, k)
        assert (row[valid:] == -1).all()
        sel = row[:valid]
        assert (sel >= 0).all() and (sel < n).all()
        assert len(set(sel.tolist())) == valid
        if w["sorted_index"]:
            assert (np.diff(sel) > 0).all()
        assert (bits[r, :valid] == x[r, sel].astype(np.uint32)).all()
        if n > k:
            mask = np.zeros(n, bool)
            mask[sel] = True
            sv, uv = vals[r, :n][mask], vals[r, :n][~mask]
            assert sv.min() >= uv.max()
            t = sv.min()
            tie_sel = np.nonzero(mask & (vals[r, :n] == t))[0]
            tie_all = np.nonzero(vals[r, :n] == t)[0]
            assert (tie_sel == tie_all[:len(tie_sel)]).all()  # a prefix in index order


@pytest.mark.parametrize("name", syn.WORKLOADS)
def test_invariants_on_workload_samples(name):
    w = syn.workload(name)
    rows = np.unique(np.linspace(0, w["rows"] - 1, 12).astype(np.int64))
    if w["nan_at"] is not None:
        rows = np.unique(np.append(rows, w["nan_at"][0]))
    s = syn.row_subset(w, rows)
    idx, bits, nan = oracle.topk(s["x"], s["dtype"], s["k"], row_end=s["row_end"],
                                 sorted_index=s["sorted_index"], cols=s["cols"])
    check_invariants(s, idx, bits, nan)
    if w["nan_at"] is not None:
        where = int(np.nonzero(rows == w["nan_at"][0])[0][0])
        assert nan[where] == 1 and nan.sum() == 1
    else:
        assert nan.sum() == 0


def test_workload_recipes():
    w = syn.workload("indexer_bf16_4096x2048_causal_k512_gather")
    assert w["row_end"][0] == 1 and w["row_end"][1023] == 512 and w["row_end"][1024] == 513
    assert w["row_end"][-1] == 2048 and (w["row_end"] <= w["k"]).sum() == 1024
    w5 = syn.workload("indexer_bf16_3x4096x16384_levels64_k2048_gather", rows=64)
    vals = oracle.bits_to_values(w5["x"], "bf16")
    lv = np.unique(vals)
    assert len(lv) <= 64 and np.all((lv * 16) % 2 == 1) and lv.min() >= -3.9375 and lv.max() <= 3.9375
    w3 = syn.workload("indexer_bf16_4x204800_k1024", rows=1)
    assert (w3["stride"] * 2) % 128 == 0


# --------------------------------------------------------------------------
# the DeepSelect tutorial's example calls (shapes and the end bound)
# --------------------------------------------------------------------------

def test_tutorial_examples():
    with open(os.path.join(GOLDEN, "deepselect_examples.json")) as f:
        g = json.load(f)
    ex = g["examples"]
    a = ex[0]
    x = syn.normal_rows(42, a["batch_size"], a["vocab_size"], a["dtype"])
    idx, bits, _ = oracle.topk(x, a["dtype"], a["topk"], sorted_index=a["sorted_index"])
    assert list(idx.shape) == a["expect_indices_shape"] and list(bits.shape) == a["expect_values_shape"]
    assert (np.diff(idx, axis=1) > 0).all()
    b = ex[1]
    x = syn.normal_rows(43, b["batch_size"], b["vocab_size"], b["dtype"])
    end = np.array(b["end"], dtype=np.int32)
    idx, _, _ = oracle.topk(x, b["dtype"], b["topk"], row_end=end, sorted_index=b["sorted_index"])
    assert list(idx.shape) == b["expect_indices_shape"]
    assert idx[1].max() < b["end"][1] and idx[0].max() < b["end"][0]
    # the end-bounded row equals top-k of the truncated row
    idx_t, _, _ = oracle.topk(np.ascontiguousarray(x[1:2, :b["end"][1]]), b["dtype"], b["topk"], sorted_index=True)
    assert (idx[1] == idx_t[0]).all()
    assert g["limits"]["max_topk"] == 4096


# --------------------------------------------------------------------------
# gather oracle: the pull request's identity and its unit-test list
# --------------------------------------------------------------------------

def advanced_index_gather(key, idx, b):
    rows, n = idx.shape
    batch = (np.arange(rows) // (rows // b))[:, None].repeat(n, axis=1)
    safe = np.maximum(idx, 0)
    return key[batch, safe]


@pytest.mark.parametrize("b", [1, 3])
def test_gather_matches_advanced_indexing_and_index_select(b):
    rng = np.random.default_rng(21 + b)
    comp_len, d, rows_per_b, n = 64, 16, 5, 9
    key = bf16bits(rng.standard_normal((b, comp_len, d)).astype(np.float32)).reshape(b, comp_len, d)
    idx = rng.integers(-1, comp_len, size=(b * rows_per_b, n)).astype(np.int64)
    out, bad = oracle.gather_rows(key, idx, b)
    assert bad == 0
    assert (out == advanced_index_gather(key, idx, b)).all()
    flat = torch.from_numpy(key.astype(np.int32).reshape(b * comp_len, d))
    batch = torch.arange(b * rows_per_b)[:, None] // rows_per_b
    pos = batch * comp_len + torch.from_numpy(np.maximum(idx, 0))
    sel = torch.index_select(flat, 0, pos.reshape(-1)).reshape(b * rows_per_b, n, d)
    assert (out.astype(np.int32) == sel.numpy()).all()


def test_gather_batches_do_not_mix():
    b, comp_len, d = 3, 8, 8
    key = np.zeros((b, comp_len, d), dtype=np.uint16)
    for bb in range(b):
        key[bb] = bb + 1
    idx = np.tile(np.arange(comp_len, dtype=np.int64), (b * 2, 1))
    out, _ = oracle.gather_rows(key, idx, b)
    for r in range(b * 2):
        assert (out[r] == r // 2 + 1).all()


def test_gather_noncontiguous_key_repeats_and_out_of_range():
    rng = np.random.default_rng(4)
    base = bf16bits(rng.standard_normal((2, 20, 48)).astype(np.float32)).reshape(2, 20, 48)
    key = base[:, :, 8:40]  # row stride 48 > d = 32
    assert not key.flags["C_CONTIGUOUS"]
    idx = np.array([[3, 3, 3, -1], [19, 0, 20, 5]], dtype=np.int64)
    out, bad = oracle.gather_rows(key, idx, 2)
    assert bad == 1
    assert (out[0, 0] == key[0, 3]).all() and (out[0, 1] == out[0, 2]).all()
    assert (out[0, 3] == key[0, 0]).all()
    assert (out[1, 0] == key[1, 19]).all() and (out[1, 2] == 0).all() and (out[1, 3] == key[1, 5]).all()


# --------------------------------------------------------------------------
# mutation checks: each planted mistake in a copy of ref.c fails a pin
# --------------------------------------------------------------------------

MUTATIONS = {
    "tie_rule_flipped": ("if (p->i < q->i) return -1;\n    if (p->i > q->i) return 1;\n    return 0;",
                         "if (p->i > q->i) return -1;\n    if (p->i < q->i) return 1;\n    return 0;"),
    "smallest_instead_of_largest": ("if (p->v > q->v) return -1;\n    if (p->v < q->v) return 1;",
                                    "if (p->v < q->v) return -1;\n    if (p->v > q->v) return 1;"),
    "row_end_off_by_one": ("n = row_end[r];", "n = row_end[r] + 1;"),
    "short_row_boundary": ("if (n <= k) {", "if (n < k) {"),
    "value_order_nan_last": ("if (pn != qn) return pn ? -1 : 1;", "if (pn != qn) return pn ? 1 : -1;"),
    "value_order_ascending": ("        if (p->v > q->v) return -1;\n        if (p->v < q->v) return 1;",
                              "        if (p->v < q->v) return -1;\n        if (p->v > q->v) return 1;"),
    "value_order_ties_flipped": ("return p->i < q->i ? -1 : (p->i > q->i);", "return p->i > q->i ? -1 : (p->i < q->i);"),
    "value_order_short_rows_by_index": ("if (sorted_index == 2)", "if (sorted_index == 3)"),
}


def _mutant_topk(src_text, tmp_path, name):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src_text)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c)])
    lib = ctypes.CDLL(str(so))
    vp, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_topk.argtypes = [vp, c_int, i64, i64, i64, vp, i64, c_int, vp, vp, vp]
    return lib


def _pins_pass(lib):
    """A compact re-run of the brute-force pin (row_end variants, ties) against a given library."""
    rng = np.random.default_rng(99)
    for kind in ("small_ints", "two_level", "normal"):
        for n in (5, 9, 16):
            x = tiny_row(kind, n, rng, "f32")[None, :].copy()
            vals = oracle.bits_to_values(x[0], "f32")
            for k in range(1, n + 2):
                for re_val in (n, n - 1):
                    re_arr = np.array([re_val], np.int32)
                    idx = np.empty((1, k), np.int64)
                    bits = np.empty((1, k), np.uint32)
                    nan = np.empty((1,), np.int32)
                    lib.oracle_topk(x.ctypes.data, 0, 1, n, n, re_arr.ctypes.data, k, 1,
                                    idx.ctypes.data, bits.ctypes.data, nan.ctypes.data)
                    want = oracle.brute_topk_row(vals, re_val, k)
                    got = [int(i) for i in idx[0] if i >= 0]
                    if got != want:
                        return False
                    if any(int(i) != -1 for i in idx[0][len(want):]):
                        return False
    # "NaN handling": a row whose valid length equals k is not checked, and a
    # short row lists its columns in order even when unsorted output is asked for
    v = np.array([3.0, np.nan, 1.0, 2.0], dtype=np.float32)
    x = f32bits(v)[None, :].copy()
    idx = np.empty((1, 4), np.int64)
    bits = np.empty((1, 4), np.uint32)
    nan = np.empty((1,), np.int32)
    lib.oracle_topk(x.ctypes.data, 0, 1, 4, 4, None, 4, 0, idx.ctypes.data, bits.ctypes.data,
                    nan.ctypes.data)
    if nan[0] != 0 or idx[0].tolist() != [0, 1, 2, 3]:
        return False
    # value order against a stable descending torch.sort: long and short rows with ties, -0/+0,
    # and a short row holding NaNs
    rows = [tiny_row(kind, 12, rng, "f32") for kind in ("small_ints", "two_level", "normal")]
    rows.append(np.array([0.0, -0.0, 1.0, -0.0, 0.0, 1.0], np.float32))
    rows.append(np.array([np.nan, 1.0, np.nan, 2.0, -np.inf, 2.0], np.float32))
    for v in rows:
        n = len(v)
        x = f32bits(v)[None, :].copy()
        has_nan = bool(np.isnan(v).any())
        for k in range(n if has_nan else 1, n + 2):
            idx = np.empty((1, k), np.int64)
            bits = np.empty((1, k), np.uint32)
            nan = np.empty((1,), np.int32)
            lib.oracle_topk(x.ctypes.data, 0, 1, n, n, None, k, 2, idx.ctypes.data, bits.ctypes.data,
                            nan.ctypes.data)
            if idx[0].tolist() != stable_sort_order(v, n, k):
                return False
    return True


def test_mutants_fail_the_pins(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ref.c")).read()
    assert _pins_pass(_mutant_topk(src, tmp_path, "unmodified"))
    for name, (old, new) in MUTATIONS.items():
        assert old in src, name
        lib = _mutant_topk(src.replace(old, new, 1), tmp_path, name)
        assert not _pins_pass(lib), f"planted mistake '{name}' went unnoticed"
