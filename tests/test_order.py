"""Value-ordered output (``sorted_value``): each row's k entries by value
descending, equal values by index ascending, fills last, a NaN of a short row
above every number.  Checked element by element against the oracle's value
order, for every selection kernel the plan can pick, and at the workloads'
full sizes on sampled rows plus a property check of every row."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import IDX_DTYPE, to_bits, to_torch
from tests.test_topk import SAMPLES, make_case, n_valid_tensor, sample_rows

pytestmark = pytest.mark.gpu


def run_value_order(w, idx_dtype="i32", want_values=True, x=None):
    import gather_radix_select_gb300 as g
    if x is None:
        x = to_torch(w["x"], w["dtype"])[:, :w["cols"]]
    end = None if w["row_end"] is None else torch.from_numpy(w["row_end"]).cuda()
    nan = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx = g.topk(x, w["k"], end=end, sorted_value=True, indices_type=IDX_DTYPE[idx_dtype],
                       return_value=want_values, nan_flag=nan, err_flag=err)
    torch.cuda.synchronize()
    return x, vals, idx, int(nan.item()), int(err.item())


def check_rows(w, rows, gpu_idx, gpu_bits):
    """GPU rows (given by ``rows``) equal the oracle's value order exactly; NaN rows are skipped."""
    s = syn.row_subset(w, rows)
    o_idx, o_bits, o_nan = oracle.topk(s["x"], w["dtype"], w["k"], row_end=s["row_end"], cols=w["cols"],
                                       sorted_value=True)
    checked = 0
    for i, r in enumerate(rows):
        if o_nan[i]:
            continue
        assert (np.asarray(gpu_idx[i], np.int64) == o_idx[i]).all(), "row %d: value order differs" % r
        if gpu_bits is not None:
            assert (np.asarray(gpu_bits[i]).astype(np.uint32) == o_bits[i]).all(), "row %d: values differ" % r
        checked += 1
    return checked


def case(dtype, rows, cols, k, kind, row_end=None):
    seed = zlib.crc32(repr(("order", dtype, rows, cols, k, kind)).encode())
    e = syn.elem_bytes(dtype)
    stride = (cols * e + 15) // 16 * 16 // e
    return make_case(dtype, rows, cols, k, kind, seed, stride=stride, row_end=row_end, sorted_index=False)


# (plan, dtype, rows, cols, k, kind): shapes each kernel takes when forced
KERNEL_CASES = [
    ("reg", "bf16", 4, 8191, 2048, "levels"),
    ("reg", "f32", 3, 4093, 4000, "zeros_inf"),
    ("reg", "f32", 5, 1021, 64, "two_level"),
    # register tiles of 2 and 8 vectors at k = 8 entries a thread (ranked inside the register
    # kernel when the call also gathers)
    ("reg", "bf16", 80, 2048, 512, "levels"),
    ("reg", "f32", 40, 3000, 1024, "normal"),
    ("row", "bf16", 5, 16384, 2048, "levels"),
    ("row", "f32", 4, 8192, 64, "normal"),
    ("row", "f32", 3, 12000, 4096, "zeros_inf"),
    # ranked inside the row kernel: the list overflows on equal rows (full-slice path), 128-thread
    # CTAs, and short bf16 rows on 256 histogram bins just inside and past the 2 * bins slot limit
    ("row", "bf16", 3, 6000, 1000, "equal"),
    ("row", "f32", 4, 4000, 1000, "two_level"),
    ("row", "bf16", 3, 4000, 512, "levels"),
    ("row", "bf16", 3, 4000, 600, "levels"),
    ("wide", "f32", 3, 131075, 4096, "normal"),
    ("wide", "bf16", 2, 204803, 1024, "levels"),
    # one CTA per row (rows >= half the SMs), ranked by the ordering launch
    ("wide", "f32", 80, 9000, 1000, "two_level"),
    ("wide", "bf16", 80, 20000, 4096, "levels"),
    ("wide", "f32", 78, 12000, 4096, "equal"),
    ("split", "bf16", 3, 100000, 3000, "zeros_inf"),
    ("split", "f32", 2, 70001, 1000, "equal"),
    ("stream", "f32", 2, 100003, 4096, "two_level"),
    ("stream", "bf16", 2, 70000, 700, "descending"),
]


@pytest.mark.parametrize("c", KERNEL_CASES, ids=lambda c: "-".join(map(str, c)))
def test_value_order_each_kernel(c, tuning):
    plan, dtype, rows, cols, k, kind = c
    tuning(plan=plan)
    w = case(dtype, rows, cols, k, kind)
    for idx_dtype, want_values in (("i32", True), ("i64", False)):
        x, vals, idx, nan, err = run_value_order(w, idx_dtype, want_values)
        assert err == 0 and nan == 0
        gb = None if vals is None else to_bits(vals)
        assert check_rows(w, np.arange(rows), idx.cpu().numpy(), gb) == rows


@pytest.mark.parametrize("plan", [None, "row"])
def test_value_order_short_rows_nan_and_signed_zero(plan, tuning):
    # rows shorter than k are ordered by value too; they are not checked for NaN, and a NaN there
    # ranks above every number; -0 and +0 tie and go by index (plan "row": ranked in the row kernel)
    if plan:
        tuning(plan=plan)
    rows, cols, k = 6, 300, 512
    g = np.random.default_rng(5)
    v = g.choice(np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 0.5], np.float32), size=(rows, cols))
    v[1, 7] = np.nan
    v[1, 3] = -np.nan
    v[4, 0] = np.nan
    for dtype in ("f32", "bf16"):
        bits = syn.f32_to_bits(v) if dtype == "f32" else syn.f32_to_bf16_bits(v)
        e = syn.elem_bytes(dtype)
        stride = (cols * e + 15) // 16 * 16 // e
        full = np.zeros((rows, stride), dtype=bits.dtype)
        full[:, :cols] = bits
        end = np.array([300, 299, 0, 1, 17, 200], np.int32)
        w = {"name": "short", "x": full, "dtype": dtype, "rows": rows, "cols": cols, "stride": stride, "k": k,
             "row_end": end, "sorted_index": False, "idx_dtype": "i32", "want_values": True, "nan_at": None}
        x, vals, idx, nan, err = run_value_order(w)
        assert err == 0 and nan == 0
        assert check_rows(w, np.arange(rows), idx.cpu().numpy(), to_bits(vals)) == rows


@pytest.mark.parametrize("plan", ["wide", "row", None])
def test_value_order_rows_with_ends(plan, tuning):
    # rows shorter than k (fills last), rows just longer, full rows, under each plan's own ranking
    if plan:
        tuning(plan=plan)
    rows, cols, k = 96, 6000, 700
    end = np.array([[0, 1, 699, 700, 701, 2500, 6000, 123][i % 8] for i in range(rows)], np.int32)
    for dtype in ("f32", "bf16"):
        w = case(dtype, rows, cols, k, "two_level", row_end=end)
        for idx_dtype, want_values in (("i32", True), ("i64", False)):
            x, vals, idx, nan, err = run_value_order(w, idx_dtype, want_values)
            assert err == 0 and nan == 0
            gb = None if vals is None else to_bits(vals)
            assert check_rows(w, np.arange(rows), idx.cpu().numpy(), gb) == rows


def test_value_order_k_one_and_k_equal_cols():
    for dtype, rows, cols, k in (("f32", 7, 5000, 1), ("bf16", 5, 4096, 4096), ("f32", 3, 64, 64)):
        w = case(dtype, rows, cols, k, "levels")
        x, vals, idx, nan, err = run_value_order(w)
        assert err == 0 and nan == 0
        assert check_rows(w, np.arange(rows), idx.cpu().numpy(), to_bits(vals)) == rows


def check_order_on_device(x, n_valid, k, idx, idx_sorted, skip_rows=()):
    """Every row of a value-ordered result holds the index-ordered result's set, values
    non-increasing, equal values by ascending index."""
    R = x.shape[0]
    keep = torch.ones(R, dtype=torch.bool, device=x.device)
    for r in skip_rows:
        keep[r] = False
    ii = idx.to(torch.int64)[keep]
    assert bool((torch.sort(torch.where(ii < 0, torch.full_like(ii, 1 << 40), ii), dim=1).values
                 == torch.where(idx_sorted.to(torch.int64)[keep] < 0, torch.full_like(ii, 1 << 40),
                                idx_sorted.to(torch.int64)[keep])).all()), "value order lost entries"
    v = torch.gather(x.float()[keep], 1, ii.clamp(min=0))
    m = torch.minimum(n_valid[keep], torch.tensor(k, device=x.device))[:, None]
    pair = torch.arange(1, k, device=x.device)[None, :] < m
    a, b = v[:, :-1], v[:, 1:]
    ok = (a > b) | ((a == b) & (ii[:, :-1] < ii[:, 1:]))
    assert bool((ok | ~pair).all()), "row not in value order"


@pytest.mark.parametrize("name", syn.WORKLOADS)
def test_value_order_workloads(name):
    import gather_radix_select_gb300 as g
    w = syn.workload(name)
    x, vals, idx, nan, err = run_value_order(w, w["idx_dtype"], w["want_values"])
    assert err == 0
    nan_rows = () if w["nan_at"] is None else (w["nan_at"][0],)
    end = None if w["row_end"] is None else torch.from_numpy(w["row_end"]).cuda()
    _, idx_sorted = g.topk(x, w["k"], end=end, sorted_index=True, indices_type=IDX_DTYPE[w["idx_dtype"]],
                           return_value=False)
    check_order_on_device(x, n_valid_tensor(w), w["k"], idx, idx_sorted, skip_rows=nan_rows)
    rows = sample_rows(w, min(SAMPLES[name], 16), nan_rows)
    gb = None if vals is None else to_bits(vals)[rows]
    assert check_rows(w, rows, idx.cpu().numpy()[rows], gb) >= len(rows) - len(nan_rows)


def test_value_order_gather_takes_the_largest():
    # with value order the gather takes the n_gather largest values' rows
    import gather_radix_select_gb300 as g
    rows, cols, k, n_gather, b, d = 64, 2048, 512, 100, 2, 128
    end = np.minimum(cols, np.arange(rows) * 40 + 1).astype(np.int32)
    w = case("bf16", rows, cols, k, "levels", row_end=end)
    x = to_torch(w["x"], "bf16")[:, :cols]
    key_bits = syn.f32_to_bf16_bits(np.random.default_rng(9).standard_normal((b, cols, d)).astype(np.float32))
    key = to_torch(key_bits.reshape(b * cols, d), "bf16").view(b, cols, d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for return_indices in (True, False):
        vals, idx, out = g.topk_gather(x, k, key, n_gather, end=torch.from_numpy(end).cuda(), sorted_value=True,
                                       return_value=True, return_indices=return_indices, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        o_idx, o_bits, _ = oracle.topk(w["x"], "bf16", k, row_end=end, cols=cols, sorted_value=True)
        if return_indices:
            assert (idx.cpu().numpy().astype(np.int64) == o_idx).all()
        else:
            assert idx is None
        assert (to_bits(vals).astype(np.uint32) == o_bits).all()
        want, bad = oracle.gather_rows(key_bits, o_idx[:, :n_gather], b=b)
        assert bad == 0
        assert (to_bits(out) == want).all()


@pytest.mark.parametrize("plan", [None, "row", "reg"])
@pytest.mark.parametrize("dtype,k,n_gather,d,b,idx_dtype,want_values", [
    ("bf16", 512, 512, 24, 3, "i32", False),    # every ordered position, 3-vector key rows
    ("bf16", 2048, 37, 128, 1, "i64", False),
    ("f32", 4096, 1000, 64, 2, "i64", True),
    ("f32", 100, 1, 8, 2, "i32", False),        # one-vector key rows, 32-thread ordering CTAs
])
def test_value_order_gather_in_the_ordering_launch(dtype, k, n_gather, d, b, idx_dtype, want_values, plan, tuning):
    # the first n_gather ordered positions' key rows are gathered (by the ordering launch, or by a
    # row or register kernel that ranks its own outputs where it can): equal to
    # torch.index_select over the batch-flattened key at the ordered indices (fills read row 0), and
    # the order itself equals the oracle's
    import gather_radix_select_gb300 as g
    if plan:
        tuning(plan=plan)
    rows_per_batch, cols = 40, 4500
    rows = b * rows_per_batch
    end = np.where(np.arange(rows) % 5 == 0, k // 2 + 1, cols - (np.arange(rows) * 97) % 300).astype(np.int32)
    w = case(dtype, rows, cols, k, "levels" if dtype == "bf16" else "normal", row_end=end)
    x = to_torch(w["x"], dtype)[:, :cols]
    key_bits = syn.f32_to_bf16_bits(np.random.default_rng(k + d).standard_normal((b, cols, d)).astype(np.float32))
    key = to_torch(key_bits.reshape(b * cols, d), "bf16").view(b, cols, d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx, out = g.topk_gather(x, k, key, n_gather, end=torch.from_numpy(end).cuda(), sorted_value=True,
                                   return_value=want_values, indices_type=IDX_DTYPE[idx_dtype], err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_idx, o_bits, _ = oracle.topk(w["x"], dtype, k, row_end=end, cols=cols, sorted_value=True)
    assert (idx.cpu().numpy().astype(np.int64) == o_idx).all()
    if want_values:
        assert (to_bits(vals).astype(np.uint32) == o_bits).all()
    sel = idx[:, :n_gather].to(torch.int64).clamp(min=0)
    batch = torch.arange(rows, device="cuda")[:, None] // rows_per_batch
    ref = torch.index_select(key.reshape(-1, d), 0, (batch * cols + sel).reshape(-1)).reshape(out.shape)
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))
    for bb in range(b):  # and the oracle's gather on sampled rows of every batch
        rr = np.array([bb * rows_per_batch, bb * rows_per_batch + 7, (bb + 1) * rows_per_batch - 1])
        want, bad = oracle.gather_rows(np.ascontiguousarray(key_bits[bb:bb + 1]), o_idx[rr][:, :n_gather], 1)
        assert bad == 0 and (to_bits(out[torch.from_numpy(rr).cuda()]) == want).all()


def test_value_order_gather_flags_positions_past_the_key():
    # a key shorter than the rows: ordered positions at or past comp_len gather a zero row and raise
    # SEL_EINVAL, as the fused and the separate gather do
    import gather_radix_select_gb300 as g
    rows, cols, k, n_gather, comp_len, d = 16, 1000, 64, 64, 600, 16
    w = case("bf16", rows, cols, k, "normal")
    x = to_torch(w["x"], "bf16")[:, :cols]
    key_bits = syn.f32_to_bf16_bits(np.random.default_rng(5).standard_normal((1, comp_len, d)).astype(np.float32))
    key = to_torch(key_bits.reshape(comp_len, d), "bf16").view(1, comp_len, d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, idx, out = g.topk_gather(x, k, key, n_gather, sorted_value=True, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    past = (idx >= comp_len).cpu()
    assert past.any()
    o = out.cpu().view(torch.int16)
    assert (o[past] == 0).all()
    ref = torch.index_select(key.reshape(-1, d), 0, idx.to(torch.int64).clamp(0, comp_len - 1).reshape(-1)).reshape(out.shape)
    assert torch.equal(o[~past], ref.cpu().view(torch.int16)[~past])


def test_value_order_rejects_both_orders():
    import gather_radix_select_gb300 as g
    x = torch.zeros((2, 64), device="cuda")
    with pytest.raises(ValueError):
        g.topk(x, 4, sorted_index=True, sorted_value=True)
