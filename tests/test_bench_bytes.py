"""bench.py's algorithmic-byte arithmetic on a hand-worked workload (no GPU)."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def tiny(dtype="bf16", idx_dtype="i32", want_values=False, key=True):
    w = {"dtype": dtype, "rows": 3, "cols": 10, "k": 4, "row_end": np.array([10, 3, 4], np.int32),
         "idx_dtype": idx_dtype, "want_values": want_values}
    if key:
        w.update(key=np.zeros((1, 5, 8), np.uint16), b=1, comp_len=5, d=8, n_gather=2)
    return w


def test_topk_bytes_read_only_rows_longer_than_k():
    import bench
    # only row 0 (10 valid > k = 4) is read: 10 x 2 bytes; every row writes 4 int32 indices
    assert bench.topk_bytes(tiny()) == 10 * 2 + 3 * 4 * 4
    # int64 indices and fp32 values: 10 x 4 read, 3 x 4 x (8 + 4) written
    assert bench.topk_bytes(tiny("f32", "i64", True)) == 10 * 4 + 3 * 4 * (8 + 4)
    # row_end absent: every row has 10 > 4 valid columns
    w = tiny()
    w["row_end"] = None
    assert bench.topk_bytes(w) == 3 * 10 * 2 + 3 * 4 * 4


def test_gather_and_step_bytes():
    import bench
    w = tiny()
    key, out = 5 * 8 * 2, 3 * 2 * 8 * 2
    assert bench.gather_bytes(w, fused=True) == key + out
    assert bench.gather_bytes(w, fused=False) == key + out + 3 * 2 * 4
    assert bench.step_bytes(w) == bench.topk_bytes(w) + key + out
    assert bench.gather_bytes(tiny(key=False), fused=True) == 0


@pytest.mark.parametrize("name", ["indexer_bf16_4096x2048_causal_k512_gather", "sampling_f32_256x131072_k4096_nan",
                                  "indexer_bf16_3x4096x16384_levels64_k2048_gather", "sampling_f32_4x8192_k64"])
def test_e2e_pieces_cover_the_rows_and_respect_key_batches(name):
    import bench
    import synthetic as syn
    w = syn.workload(name)
    pieces = bench.e2e_pieces(w, 4)
    assert pieces[0][0] == 0 and pieces[-1][1] == w["rows"]
    assert all(pieces[i][1] == pieces[i + 1][0] for i in range(len(pieces) - 1))
    if w.get("key") is not None:
        rpb = w["rows_per_batch"]
        for s, e, b0, b1 in pieces:
            assert b0 * rpb <= s < e <= b1 * rpb
            assert b1 - b0 == 1 or (s == b0 * rpb and e == b1 * rpb)
