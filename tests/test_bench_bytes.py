"""bench.py's algorithmic-byte arithmetic on a hand-worked workload (no GPU)."""
import os
import sys

import numpy as np

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
