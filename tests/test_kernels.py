"""Each selection kernel, forced with SEL_PLAN, against the oracle on every row.

The automatic plan sends a shape to one kernel; these cases force the
others onto the same shapes so that every kernel's paths run: several ring
chunks with a ragged tail, a ring that holds the whole row, threshold
estimates that keep too few or too many keys (sorted rows, constant rows),
ties, infinities, variable row ends, NaN rows and the fused gather.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import compare_with_oracle, to_bits, to_torch
from tests.test_topk import make_case, run

pytestmark = pytest.mark.gpu

CASES = [
    # (dtype, rows, cols, k, kind)
    ("f32", 3, 70001, 1000, "normal"),
    ("bf16", 2, 204803, 1024, "normal"),
    ("f32", 2, 20000, 300, "normal"),
    ("bf16", 3, 100000, 4096, "ascending"),
    ("bf16", 3, 100000, 4096, "descending"),
    ("f32", 2, 100000, 64, "equal"),
    ("f32", 2, 100003, 4096, "zeros_inf"),
    ("bf16", 5, 70000, 700, "levels"),
    ("f32", 4, 131072, 4096, "normal"),
]

MODES = ["wide", "split", "stream", "flat"]

# shapes the register-resident kernel holds (bf16 up to 32768 columns, fp32 up to 16384): every
# tile size, ragged tails ending inside a vector, ties, infinities and near-full selections
REG_CASES = [
    ("bf16", 5, 2000, 512, "normal"),
    ("bf16", 3, 2047, 700, "levels"),
    ("f32", 4, 1021, 300, "zeros_inf"),
    ("f32", 3, 4093, 4000, "normal"),
    ("bf16", 4, 8191, 2048, "levels"),
    ("f32", 2, 16384, 4096, "two_level"),
    ("bf16", 3, 16383, 64, "equal"),
    ("bf16", 2, 32768, 4096, "ascending"),
    ("f32", 3, 9999, 1, "descending"),
]


@pytest.mark.parametrize("case", REG_CASES, ids=lambda c: "-".join(map(str, c)))
def test_reg_kernel(case, tuning):
    tuning(plan="reg")
    import gather_radix_select_gb300 as g
    dtype, rows, cols, k, kind = case
    assert g.kernel_name(torch.float32 if dtype == "f32" else torch.bfloat16, rows, cols, k) == "reg_kernel"
    w = padded(*case)
    x, end, vals, idx, nan, err = run(w)
    assert err == 0 and nan == 0
    compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), to_bits(vals), True)
    x, end, vals, idx, nan, err = run(w, sorted_index=False, idx_dtype="i64", want_values=False)
    assert err == 0
    compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), None, False)


def padded(dtype, rows, cols, k, kind, row_end=None):
    seed = zlib.crc32(repr((dtype, rows, cols, k, kind)).encode())
    e = syn.elem_bytes(dtype)
    stride = (cols * e + 15) // 16 * 16 // e
    return make_case(dtype, rows, cols, k, kind, seed, stride=stride, row_end=row_end)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_forced_kernel(mode, case, tuning):
    tuning(plan=mode)
    dtype, rows, cols, k, kind = case
    w = padded(*case)
    x, end, vals, idx, nan, err = run(w)
    assert err == 0 and nan == 0
    compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), to_bits(vals), True)
    x, end, vals, idx, nan, err = run(w, sorted_index=False, idx_dtype="i64", want_values=False)
    assert err == 0
    compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), None, False)


@pytest.mark.parametrize("parts", ["1", "2", "7", "64"])
def test_wide_parts(parts, tuning):
    # the streaming kernel on one CTA per row, and with rows split over CTAs whose candidate lists
    # meet in the workspace (the last part to arrive merges)
    tuning(plan="wide")
    tuning(parts=int(parts))
    for case in (("f32", 3, 131075, 4096, "normal"), ("bf16", 2, 204803, 1024, "levels"),
                 ("f32", 2, 70001, 100, "descending"), ("bf16", 3, 100000, 3000, "zeros_inf")):
        w = padded(*case)
        x, end, vals, idx, nan, err = run(w)
        assert err == 0 and nan == 0
        compare_with_oracle(w, np.arange(case[1]), idx.cpu().numpy(), to_bits(vals), True)


# shapes for the per-warp candidate regions of the streaming kernel: thresholds at or below zero
# (raw-bit compare not usable), rows shorter than one 16-byte vector, ragged tails, candidates
# piling into one warp's range, and a row whose every element ties
WIDE_CASES = [
    ("f32", 3, 5000, 4096, "normal"),
    ("bf16", 2, 3000, 2999, "normal"),
    ("f32", 4, 3, 1, "normal"),
    ("bf16", 4, 7, 2, "normal"),
    ("bf16", 3, 100007, 333, "zeros_inf"),
    ("f32", 2, 66001, 4096, "ascending"),
    ("bf16", 2, 70000, 1000, "equal"),
    ("f32", 2, 131072, 4096, "two_level"),
]


@pytest.mark.parametrize("case", WIDE_CASES, ids=lambda c: "-".join(map(str, c)))
def test_wide_kernel_paths(case, tuning):
    tuning(plan="wide")
    w = padded(*case)
    x, end, vals, idx, nan, err = run(w)
    assert err == 0 and nan == 0
    compare_with_oracle(w, np.arange(case[1]), idx.cpu().numpy(), to_bits(vals), True)
    x, end, vals, idx, nan, err = run(w, sorted_index=False, idx_dtype="i64", want_values=False)
    assert err == 0
    compare_with_oracle(w, np.arange(case[1]), idx.cpu().numpy(), None, False)


@pytest.mark.parametrize("mode", MODES + ["reg"])
def test_forced_row_end_and_nan(mode, tuning):
    tuning(plan=mode)
    rows, cols, k = 6, (12000 if mode == "reg" else 90000), 2000
    row_end = np.array([0, 1999, 2000, 2001, cols // 2, 200000], dtype=np.int32)
    w = padded("f32", rows, cols, k, "normal", row_end=row_end)
    x, end, vals, idx, nan, err = run(w)
    assert err == 0 and nan == 0
    compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), to_bits(vals), True)
    # a NaN inside the valid part of a long row raises the flag; one past row_end does not
    bits = w["x"].copy()
    bits[4, cols // 2 + 5] = 0x7FC00000  # beyond row_end[4]: ignored
    w2 = dict(w, x=bits)
    _, _, _, _, nan, err = run(w2)
    assert err == 0 and nan == 0
    bits[5, cols - 100] = 0xFFC00000  # a negative NaN
    w3 = dict(w, x=bits)
    _, _, vals, idx, nan, err = run(w3)
    assert err == 0 and nan == 1
    compare_with_oracle(w3, np.arange(5), idx.cpu().numpy()[:5], to_bits(vals)[:5], True)


@pytest.mark.parametrize("mode", MODES + ["reg"])
def test_forced_fused_gather(mode, tuning):
    tuning(plan=mode)
    import gather_radix_select_gb300 as g
    rng = np.random.default_rng(5)
    b, rows, cols, k, ng, d = 2, 4, (30000 if mode == "reg" else 150000), 1024, 700, 64
    v = rng.standard_normal((rows, cols)).astype(np.float32)
    x = to_torch(syn.f32_to_bf16_bits(v), "bf16")
    key_bits = syn.f32_to_bf16_bits(rng.standard_normal((b, cols, d)).astype(np.float32)).reshape(b, cols, d)
    key = to_torch(key_bits, "bf16")
    end = torch.from_numpy(np.array([cols, 1000, cols * 3 // 5 + 1, cols - 1], dtype=np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, fidx, fout = g.topk_gather(x, k, key, ng, end=end, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_idx, _, _ = oracle.topk(syn.f32_to_bf16_bits(v), "bf16", k, row_end=end.cpu().numpy(), sorted_index=True,
                              cols=cols)
    assert (fidx.cpu().numpy().astype(np.int64) == o_idx).all()
    want, bad = oracle.gather_rows(key_bits, o_idx[:, :ng], b)
    assert bad == 0 and (to_bits(fout) == want).all()


@pytest.mark.parametrize("mode", ["reg", "row", "wide"])
@pytest.mark.parametrize("d", [48, 200, 512, 2048])
def test_fused_gather_row_widths(mode, d, tuning):
    # key rows of 6, 25, 64 and 256 16-byte vectors: the general copy loop (not a power of two, or
    # wider than the CTA) and the per-column one; the last case has a key shorter than the scored
    # row, so some selected positions are out of range (zero rows, error flag)
    tuning(plan=mode)
    import gather_radix_select_gb300 as g
    rng = np.random.default_rng(d)
    b, rows, k, ng = 2, 6, 300, 200
    cols = {"reg": 3000, "row": 20000, "wide": 140000}[mode]
    comp_len = cols if d != 2048 else cols // 2
    v = rng.standard_normal((rows, cols)).astype(np.float32)
    x = to_torch(syn.f32_to_bf16_bits(v), "bf16")
    key_bits = syn.f32_to_bf16_bits(rng.standard_normal((b, comp_len, d)).astype(np.float32)).reshape(b, comp_len, d)
    key = to_torch(key_bits, "bf16")
    end = torch.from_numpy(np.array([cols, 200, cols // 2, cols - 1, 299, 7], dtype=np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, fidx, fout = g.topk_gather(x, k, key, ng, end=end, err_flag=err)
    torch.cuda.synchronize()
    o_idx, _, _ = oracle.topk(syn.f32_to_bf16_bits(v), "bf16", k, row_end=end.cpu().numpy(), sorted_index=True,
                              cols=cols)
    assert (fidx.cpu().numpy().astype(np.int64) == o_idx).all()
    want, bad = oracle.gather_rows(key_bits, o_idx[:, :ng], b)
    assert (to_bits(fout) == want).all()
    assert int(err.item()) == (1 if bad else 0)
    assert (bad > 0) == (d == 2048)


@pytest.mark.parametrize("mode", ["reg", "row", "wide", "split", "stream"])
def test_row_order_interleaved_and_in_order_agree(mode, tuning):
    # with per-row ends CTAs take rows from both ends of the batch alternately; the result must be
    # the same, bit for bit, as taking them in order, and equal to the oracle
    import gather_radix_select_gb300 as g
    rows, cols, k = 37, (4000 if mode == "reg" else 70000), 300
    row_end = np.minimum(cols, (np.arange(rows) * (cols // rows)) + 7).astype(np.int32)
    row_end[5] = 0
    w = padded("f32", rows, cols, k, "normal", row_end=row_end)
    res = []
    for order in (True, False):
        tuning(plan=mode, row_order=order)
        x, end, vals, idx, nan, err = run(w)
        assert err == 0 and nan == 0
        res.append((idx.cpu().numpy(), to_bits(vals)))
    assert (res[0][0] == res[1][0]).all() and (res[0][1] == res[1][1]).all()
    compare_with_oracle(w, np.arange(rows), res[0][0], res[0][1], True)
    assert g.get_tuning()["row_order"] is False
