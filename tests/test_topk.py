"""GPU parity of sel_topk (through the C ABI) against the CPU oracle.

Full-size named workloads: exact comparison with the oracle on sampled rows
and, on every row, the defining property of top-k checked on the device.
Edge shapes: exact comparison with the oracle on every row.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import (IDX_DTYPE, TORCH_DTYPE, check_definition_on_device, compare_with_oracle, to_bits,
                         to_torch)

pytestmark = pytest.mark.gpu


def gsel():
    import gather_radix_select_gb300 as g
    return g


def run(w, *, sorted_index=None, idx_dtype=None, want_values=None, x=None):
    g = gsel()
    sorted_index = w["sorted_index"] if sorted_index is None else sorted_index
    idx_dtype = w["idx_dtype"] if idx_dtype is None else idx_dtype
    want_values = w["want_values"] if want_values is None else want_values
    if x is None:
        x = to_torch(w["x"], w["dtype"])[:, :w["cols"]]
    end = None if w["row_end"] is None else torch.from_numpy(w["row_end"]).cuda()
    nan = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx = g.topk(x, w["k"], end=end, sorted_index=sorted_index, indices_type=IDX_DTYPE[idx_dtype],
                       return_value=want_values, nan_flag=nan, err_flag=err)
    torch.cuda.synchronize()
    return x, end, vals, idx, int(nan.item()), int(err.item())


def sample_rows(w, count, extra=()):
    R = w["rows"]
    rows = set(np.linspace(0, R - 1, min(count, R)).astype(np.int64).tolist())
    rows.update(int(r) for r in extra if 0 <= r < R)
    return np.array(sorted(rows), dtype=np.int64)


def n_valid_tensor(w):
    if w["row_end"] is None:
        return torch.full((w["rows"],), w["cols"], dtype=torch.int64, device="cuda")
    return torch.from_numpy(np.clip(w["row_end"], 0, w["cols"]).astype(np.int64)).cuda()


SAMPLES = {
    "sampling_f32_4x8192_k64": 4,
    "indexer_bf16_4096x2048_causal_k512_gather": 48,
    "indexer_bf16_4x204800_k1024": 4,
    "sampling_f32_256x131072_k4096_nan": 24,
    "indexer_bf16_3x4096x16384_levels64_k2048_gather": 48,
}


@pytest.mark.parametrize("name", syn.WORKLOADS)
def test_workload_parity(name):
    w = syn.workload(name)
    x, end, vals, idx, nan, err = run(w)
    assert err == 0
    nan_rows = () if w["nan_at"] is None else (w["nan_at"][0],)
    expect_nan = 0
    if w["nan_at"] is not None:
        r, c = w["nan_at"]
        n = syn_valid(w, r)
        expect_nan = int(n > w["k"] and c < n)
    assert nan == expect_nan
    extra = list(nan_rows)
    if w["row_end"] is not None:
        # rows around the short/long boundary
        re = np.clip(w["row_end"], 0, w["cols"])
        b = np.nonzero(re > w["k"])[0]
        if len(b):
            extra += [int(b[0]) - 1, int(b[0]), int(b[0]) + 1]
    rows = sample_rows(w, SAMPLES[name], extra)
    gi = idx.cpu().numpy()[rows]
    gb = None if vals is None else to_bits(vals)[rows]
    checked, _ = compare_with_oracle(w, rows, gi, gb, w["sorted_index"], skip_rows=nan_rows)
    assert checked >= len(rows) - len(nan_rows)
    check_definition_on_device(x, n_valid_tensor(w), w["k"], idx, vals, w["sorted_index"], skip_rows=nan_rows)


def syn_valid(w, r):
    if w["row_end"] is None:
        return w["cols"]
    return int(min(max(int(w["row_end"][r]), 0), w["cols"]))


@pytest.mark.parametrize("name", ["sampling_f32_4x8192_k64", "indexer_bf16_4x204800_k1024"])
def test_modes_agree(name):
    """Every (sorted, idx dtype, values) mode selects the same set."""
    w = syn.workload(name)
    base_idx = None
    for sorted_index in (True, False):
        for idx_dtype in ("i32", "i64"):
            for want_values in (True, False):
                x, end, vals, idx, nan, err = run(w, sorted_index=sorted_index, idx_dtype=idx_dtype,
                                                  want_values=want_values)
                assert err == 0
                got = np.sort(idx.cpu().numpy().astype(np.int64), axis=1)
                if base_idx is None:
                    base_idx = got
                assert (got == base_idx).all()
                rows = np.arange(w["rows"])
                gb = None if vals is None else to_bits(vals)
                compare_with_oracle(w, rows, idx.cpu().numpy(), gb, sorted_index)


def make_case(dtype, rows, cols, k, kind, seed, stride=None, row_end=None, sorted_index=True, idx_dtype="i32",
              want_values=True):
    g = np.random.default_rng(seed)
    if kind == "normal":
        v = g.standard_normal((rows, cols)).astype(np.float32)
    elif kind == "equal":
        v = np.full((rows, cols), 0.75, dtype=np.float32)
    elif kind == "two_level":
        v = np.where(g.random((rows, cols)) < 0.5, 1.0, -1.0).astype(np.float32)
    elif kind == "ascending":
        v = np.tile(np.arange(cols, dtype=np.float32), (rows, 1))
    elif kind == "descending":
        v = np.tile(-np.arange(cols, dtype=np.float32), (rows, 1))
    elif kind == "zeros_inf":
        v = g.choice(np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0], np.float32), size=(rows, cols))
    elif kind == "strided_large":
        # large values only in every 8th 16-byte vector: a strided sample of the row overestimates
        # the threshold, which must be caught and corrected
        v = g.standard_normal((rows, cols)).astype(np.float32)
        per_vec = 4 if dtype == "f32" else 8
        v[:, (np.arange(cols) // per_vec) % 8 == 0] += 100.0
    elif kind == "levels":
        v = (g.integers(0, 64, size=(rows, cols)) * 2 - 63).astype(np.float32) / 16
    else:
        raise ValueError(kind)
    bits = syn.f32_to_bits(v) if dtype == "f32" else syn.f32_to_bf16_bits(v)
    stride = cols if stride is None else stride
    if stride != cols:
        full = np.zeros((rows, stride), dtype=bits.dtype)
        full[:, :cols] = bits
        bits = full
    return {"name": "edge", "x": bits, "dtype": dtype, "rows": rows, "cols": cols, "stride": stride, "k": k,
            "row_end": row_end, "sorted_index": sorted_index, "idx_dtype": idx_dtype, "want_values": want_values,
            "nan_at": None}


EDGE = [
    # (dtype, rows, cols, k, kind)
    ("f32", 1, 1, 1, "normal"),
    ("bf16", 3, 1, 5, "normal"),
    ("f32", 5, 100, 1, "two_level"),
    ("bf16", 2, 5000, 4096, "normal"),
    ("f32", 2, 4097, 4096, "normal"),
    ("f32", 3, 64, 4096, "normal"),
    ("f32", 4, 3000, 17, "equal"),
    ("bf16", 4, 3000, 17, "equal"),
    ("f32", 2, 70000, 1000, "equal"),
    ("bf16", 2, 70000, 1000, "equal"),
    ("f32", 3, 5000, 100, "ascending"),
    ("f32", 3, 5000, 100, "descending"),
    ("bf16", 3, 40000, 2000, "ascending"),
    ("bf16", 3, 40000, 2000, "descending"),
    ("f32", 4, 999, 31, "zeros_inf"),
    ("bf16", 4, 20000, 333, "zeros_inf"),
    ("f32", 8, 16383, 700, "levels"),
    ("bf16", 8, 16385, 700, "levels"),
    ("f32", 2, 131072 * 2 + 3, 4096, "normal"),
    ("bf16", 1, 262147, 64, "normal"),
    ("f32", 300, 1000, 64, "normal"),
    ("bf16", 700, 4100, 256, "two_level"),
    # one CTA per row with a threshold bin too large for the candidate list: full-slice path
    ("bf16", 320, 16384, 100, "equal"),
    ("f32", 320, 9000, 64, "two_level"),
    ("bf16", 320, 16384, 2048, "levels"),
    ("f32", 310, 40000, 4096, "zeros_inf"),
    # sampled threshold estimate too high -> exact fallback
    ("f32", 4, 16384, 4096, "strided_large"),
    ("f32", 320, 16384, 4096, "strided_large"),
    ("bf16", 320, 32768, 4096, "strided_large"),
    ("bf16", 2, 262144, 4096, "strided_large"),
    # split rows whose per-slice estimates miss the true threshold (sorted rows)
    ("f32", 4, 70000, 1000, "ascending"),
    ("bf16", 4, 204800, 1024, "descending"),
    ("bf16", 3, 204800, 1024, "ascending"),
    # rows wider than the split plan covers: streamed passes over global memory
    ("f32", 1, 5000000, 500, "normal"),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "-".join(map(str, c)))
def test_edge_shapes(case):
    dtype, rows, cols, k, kind = case
    seed = zlib.crc32(repr(case).encode())
    e = syn.elem_bytes(dtype)
    stride = (cols * e + 15) // 16 * 16 // e
    w = make_case(dtype, rows, cols, k, kind, seed, stride=stride)
    x, end, vals, idx, nan, err = run(w)
    assert err == 0 and nan == 0
    compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), to_bits(vals), True)
    # unsorted, int64, no values
    x, end, vals, idx, nan, err = run(w, sorted_index=False, idx_dtype="i64", want_values=False)
    compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), None, False)


def test_padded_stride_is_never_read():
    # cols = 204801, stride = 204864 (a 128-byte multiple); pad columns hold +inf
    w = make_case("bf16", 2, 204801, 1024, "normal", 5, stride=204864)
    w["x"][:, 204801:] = 0x7F80
    x, end, vals, idx, nan, err = run(w)
    assert err == 0
    assert int(idx.max()) < 204801
    compare_with_oracle(w, np.arange(2), idx.cpu().numpy(), to_bits(vals), True)


def test_row_end_variants():
    rng = np.random.default_rng(77)
    for dtype, cols, k in (("f32", 9000, 700), ("bf16", 50000, 2048), ("f32", 140000, 4096)):
        rows = 40
        w = make_case(dtype, rows, cols, k, "normal", 3 + cols)
        re = rng.integers(-5, cols + 10, size=rows).astype(np.int32)
        re[:6] = [0, 1, k - 1, k, k + 1, cols]
        w["row_end"] = re
        x, end, vals, idx, nan, err = run(w)
        assert err == 0
        compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), to_bits(vals), True)
        x, end, vals, idx, nan, err = run(w, sorted_index=False, want_values=False)
        compare_with_oracle(w, np.arange(rows), idx.cpu().numpy(), None, False)


def test_nan_flag_rules():
    # "NaN handling": only rows whose valid length exceeds k are checked
    v = np.random.default_rng(1).standard_normal((4, 6000)).astype(np.float32)
    v[0, 10] = np.nan   # long row: flagged
    v[1, 5999] = np.nan  # NaN beyond row_end: not in the row
    v[2, 3] = np.nan     # short row (n <= k): not checked
    for dtype in ("f32", "bf16"):
        bits = syn.f32_to_bits(v) if dtype == "f32" else syn.f32_to_bf16_bits(v)
        base = {"name": "nan", "x": bits, "dtype": dtype, "rows": 4, "cols": 6000, "stride": 6000, "k": 100,
                "sorted_index": True, "idx_dtype": "i32", "want_values": True, "nan_at": None}
        for rows_end, expect in (([6000, 5000, 100, 6000], 1), ([50, 5000, 100, 6000], 0)):
            w = dict(base, row_end=np.array(rows_end, np.int32))
            x, end, vals, idx, nan, err = run(w)
            assert nan == expect, (dtype, rows_end)
            assert err == 0


def test_empty_and_zero_width():
    g = gsel()
    x = torch.zeros((0, 64), dtype=torch.float32, device="cuda")
    vals, idx = g.topk(x, 8)
    assert idx.shape == (0, 8)
    x = torch.zeros((3, 0), dtype=torch.bfloat16, device="cuda")
    vals, idx = g.topk(x, 4)
    torch.cuda.synchronize()
    assert (idx == -1).all()
    assert (to_bits(vals) == 0xFF80).all()


def test_k_limits_rejected():
    g = gsel()
    x = torch.zeros((2, 64), dtype=torch.float32, device="cuda")
    for k in (0, 4097):
        with pytest.raises(g.SelError):
            g.topk(x, k)


def test_misaligned_stride_rejected():
    g = gsel()
    x = torch.zeros((2, 65), dtype=torch.float32, device="cuda")  # 260-byte rows
    with pytest.raises(g.SelError) as e:
        g.topk(x, 8)
    assert e.value.status == 2


def test_stride_requirement():
    g = gsel()
    assert g.stride_requirement() == (16, 16)
    assert g.max_cols(torch.float32) >= 262147 and g.max_cols(torch.bfloat16) >= 262147


def test_output_idx_buffer_is_used():
    g = gsel()
    w = make_case("f32", 3, 5000, 100, "normal", 9)
    x = to_torch(w["x"], "f32")
    buf = torch.full((3, 128), -7, dtype=torch.int64, device="cuda")
    _, idx = g.topk(x, 100, indices_type=torch.int64, output_idx=buf, return_value=False, sorted_index=True)
    torch.cuda.synchronize()
    assert idx.data_ptr() == buf.data_ptr()
    assert (buf[:, 100:] == -7).all()
    compare_with_oracle(w, np.arange(3), buf[:, :100].cpu().numpy(), None, True)
