"""CPU oracle for row-wise top-k and the flat row gather.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
the benchmark's ``cpu_baseline`` / reference leg may import this package.
The product (``gather_radix_select_gb300``) never imports it, and the two
share no code: the oracle is plain C (``oracle/ref.c``) plus the pure-Python
brute force below, written from the definitions on the pages:

* "Speed up PyTorch TopK with DeepSelect" (tutorial) -- "Basic TopK usage",
  "Working with variable-length rows", "NaN handling", "Supported workloads";
* MindSpore hyper-parallel pull request "perf/gather-index-select" -- the
  identity key[b, pos] == index_select(key_flat, b * comp_len + pos), and the
  block-level candidate positions of its ``compressed_candidate_topk`` chain.

Every oracle function here is pinned by ``tests/test_oracle.py`` against
things other than itself (brute force, closed forms, numpy / torch CPU
routines, the pages' example shapes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")
_SRC = os.path.join(_HERE, "ref.c")

F32, BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle/ref.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
                               "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i64, i32, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
            lib.oracle_topk.argtypes = [vp, c_int, i64, i64, i64, vp, i64, c_int, vp, vp, vp]
            lib.oracle_topk.restype = c_int
            lib.oracle_gather_rows.argtypes = [vp, i64, i64, i64, i64, i64, vp, i64, i64, i64, vp]
            lib.oracle_gather_rows.restype = i64
            lib.oracle_value_fill_bits.argtypes = [c_int]
            lib.oracle_value_fill_bits.restype = ctypes.c_uint32
            _lib = lib
    return _lib


def _dtype_code(dtype: str) -> int:
    if dtype == "f32":
        return F32
    if dtype == "bf16":
        return BF16
    raise ValueError(dtype)


def value_fill_bits(dtype: str) -> int:
    return int(_load().oracle_value_fill_bits(_dtype_code(dtype)))


def topk(x_bits: np.ndarray, dtype: str, k: int, row_end=None, sorted_index: bool = False,
         cols: int | None = None, sorted_value: bool = False):
    """Row-wise top-k by full sort (value descending, smaller index first on ties).

    x_bits : uint32 (fp32) or uint16 (bf16) bit array [rows, stride]; the
             first ``cols`` columns (default: all) are data.
    Returns (idx int64 [rows, k], bits uint32 [rows, k], row_nan int32 [rows]).
    Unsorted results come in value-descending order; sorted ones by index.
    ``sorted_value``: every row (short ones too) by value descending, ties by
    index, a NaN above every number, fills last.
    """
    if sorted_index and sorted_value:
        raise ValueError("sorted_index and sorted_value exclude each other")
    x_bits = np.ascontiguousarray(x_bits)
    want = np.uint32 if dtype == "f32" else np.uint16
    if x_bits.dtype != want or x_bits.ndim != 2:
        raise TypeError("x_bits must be a 2-D %s array" % np.dtype(want).name)
    rows, stride = x_bits.shape
    cols = stride if cols is None else cols
    re = None
    if row_end is not None:
        re = np.ascontiguousarray(row_end, dtype=np.int32)
        if re.shape != (rows,):
            raise ValueError("row_end must have one entry per row")
    out_idx = np.empty((rows, k), dtype=np.int64)
    out_bits = np.empty((rows, k), dtype=np.uint32)
    row_nan = np.empty((rows,), dtype=np.int32)
    rc = _load().oracle_topk(x_bits.ctypes.data, _dtype_code(dtype), rows, cols, stride,
                             None if re is None else re.ctypes.data, k, 2 if sorted_value else int(bool(sorted_index)),
                             out_idx.ctypes.data, out_bits.ctypes.data, row_nan.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_topk rejected its arguments")
    return out_idx, out_bits, row_nan


def gather_rows(key_bits: np.ndarray, idx: np.ndarray, b: int | None = None):
    """out[r, j, :] = key[r // (rows // b), max(idx[r, j], 0), :] (zero row if idx >= comp_len).

    key_bits : uint16 [b, comp_len, d] (any strides; bf16 bit patterns)
    idx      : integer [rows, n]
    Returns (out uint16 [rows, n, d], number of out-of-range positions).
    """
    if key_bits.dtype != np.uint16 or key_bits.ndim != 3:
        raise TypeError("key_bits must be a 3-D uint16 array")
    bb, comp_len, d = key_bits.shape
    b = bb if b is None else b
    if b != bb:
        raise ValueError("b must equal key.shape[0]")
    st = key_bits.strides
    if st[2] != 2 or st[0] % 2 or st[1] % 2:
        raise ValueError("key rows must have unit element stride")
    idx64 = np.ascontiguousarray(idx, dtype=np.int64)
    rows, n = idx64.shape
    out = np.empty((rows, n, d), dtype=np.uint16)
    # pass the array's own base pointer and element strides (non-contiguous keys allowed)
    bad = _load().oracle_gather_rows(key_bits.ctypes.data, b, comp_len, d, st[0] // 2, st[1] // 2,
                                     idx64.ctypes.data, rows, n, n, out.ctypes.data)
    if bad < 0:
        raise ValueError("oracle_gather_rows rejected its arguments")
    return out, int(bad)


def block_candidates(score_bits: np.ndarray, dtype: str, topk_blocks: int, block_size: int, pos_end=None):
    """Block-level candidate positions of the ``compressed_candidate_topk`` chain
    (MindSpore hyper-parallel pull request "perf/gather-index-select": a top-k over
    blocks expanded to ``topk_blocks * block_size`` positions, then its Sort and
    MaskedFill steps), written as its definition.

    Row r has the valid positions [0, pe) with pe = clamp(pos_end[r], 0, n_blocks *
    block_size); block c covers positions [c * block_size, (c + 1) * block_size) and
    is a candidate when it holds a valid position (c * block_size < pe).  The
    ``topk_blocks`` candidates with the largest scores are chosen by ``topk``'s rule
    (smaller block first on ties; all candidates when there are fewer).  Each chosen
    block contributes its valid positions; they are listed in ascending order and
    the rest of the row is -1.

    score_bits : uint32 (fp32) / uint16 (bf16) bits [rows, n_blocks].
    Returns (positions int64 [rows, topk_blocks * block_size], row_nan int32 [rows]).
    """
    rows, n_blocks = score_bits.shape
    limit = n_blocks * block_size
    if pos_end is None:
        pe = np.full(rows, limit, dtype=np.int64)
    else:
        pe = np.clip(np.asarray(pos_end, dtype=np.int64), 0, limit)
    n_cand = (pe + block_size - 1) // block_size
    blocks, _, row_nan = topk(score_bits, dtype, topk_blocks, row_end=n_cand.astype(np.int32), sorted_index=True)
    out = np.full((rows, topk_blocks * block_size), -1, dtype=np.int64)
    for r in range(rows):
        pos = [int(c) * block_size + i for c in blocks[r] if c >= 0 for i in range(block_size)
               if int(c) * block_size + i < pe[r]]
        pos.sort()
        out[r, :len(pos)] = pos
    return out, row_nan


# --------------------------------------------------------------------------
# Brute force on tiny rows (pure Python): the rank definition of top-k
# --------------------------------------------------------------------------

def bits_to_values(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of fp32 / bf16 bit patterns (bf16 = upper half of an fp32)."""
    if dtype == "f32":
        return np.asarray(bits, dtype=np.uint32).view(np.float32).astype(np.float64)
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def brute_topk_row(values, n: int, k: int) -> list[int]:
    """Selected columns of one row by rank counting, in ascending column order.

    Column j (j < n) is selected iff fewer than k columns i < n beat it, where
    i beats j when values[i] > values[j], or values[i] == values[j] and i < j.
    For n <= k every valid column is selected.  O(n^2); tiny rows only.
    """
    vals = [float(v) for v in values[:n]]
    chosen = []
    for j in range(n):
        beaten_by = 0
        for i in range(n):
            if vals[i] > vals[j] or (vals[i] == vals[j] and i < j):
                beaten_by += 1
        if beaten_by < k:
            chosen.append(j)
    return chosen
