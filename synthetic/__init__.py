"""Seeded synthetic inputs for the row-wise top-k and the flat row gather.

This module only draws random numbers and lays them out; it holds no step of
the selection or of the gather.  Both the CPU oracle (through the tests) and
the CUDA path are fed from here, so they always see the same bytes.

Element data are carried as raw bit patterns:

* fp32 rows as ``np.uint32`` (the IEEE-754 single bits),
* bf16 rows as ``np.uint16`` (the upper half of an fp32; rounding from fp32
  to bf16 is done by ``torch.Tensor.to(torch.bfloat16)``, i.e. round to
  nearest even).

The five named workloads follow the shapes of the DeepSelect tutorial
("Speed up PyTorch TopK with DeepSelect": "Supported workloads", "Basic TopK
usage", "Working with variable-length rows", "NaN handling") and of the
MindSpore hyper-parallel pull request "perf/gather-index-select" (gather of
compressed keys, head_dim 128, compressed length 2048 / 16384).  No public
dataset is involved: every input is drawn from a fixed seed.
"""
from __future__ import annotations

import numpy as np

F32 = "f32"
BF16 = "bf16"
I32 = "i32"
I64 = "i64"

# Seed of workload N is SEED_BASE + N (N = 1..5 in the order of WORKLOADS).
SEED_BASE = 1000


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even) and return the 16-bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bits_dtype(dtype: str):
    return np.uint32 if dtype == F32 else np.uint16


def elem_bytes(dtype: str) -> int:
    return 4 if dtype == F32 else 2


# --------------------------------------------------------------------------
# Generic draws
# --------------------------------------------------------------------------

def normal_rows(seed: int, rows: int, cols: int, dtype: str, scale: float = 1.0,
                stride: int | None = None, pad_bits: int = 0) -> np.ndarray:
    """rows x stride bit array; columns [0, cols) are N(0, scale^2), the rest pad_bits."""
    stride = cols if stride is None else stride
    g = rng_for(seed)
    v = g.standard_normal((rows, cols), dtype=np.float32)
    if scale != 1.0:
        v = v * np.float32(scale)
    bits = f32_to_bits(v) if dtype == F32 else f32_to_bf16_bits(v)
    if stride == cols:
        return bits
    out = np.full((rows, stride), pad_bits, dtype=bits.dtype)
    out[:, :cols] = bits
    return out


def levels64_bf16(seed: int, rows: int, cols: int) -> np.ndarray:
    """bf16 scores quantised to 64 distinct levels (heavy ties).

    z ~ N(0,1); level = clamp(floor((z + 4) * 8), 0, 63); value = (2*level - 63)/16.
    All 64 values are odd multiples of 1/16 in [-3.9375, 3.9375], exact in bf16,
    and none is zero.
    """
    g = rng_for(seed)
    z = g.standard_normal((rows, cols), dtype=np.float32)
    lvl = np.clip(np.floor((z + np.float32(4.0)) * np.float32(8.0)), 0, 63).astype(np.int32)
    v = ((2 * lvl - 63).astype(np.float32) / np.float32(16.0))
    return f32_to_bf16_bits(v)


def causal_row_end(rows: int, cols: int) -> np.ndarray:
    """row_end[i] = min(cols, i // 2 + 1): a causal indexer at two queries per key block."""
    i = np.arange(rows, dtype=np.int64)
    return np.minimum(cols, i // 2 + 1).astype(np.int32)


def uniform_row_end(seed: int, rows: int, cols: int) -> np.ndarray:
    """row_end ~ U{1..cols}, independently per row."""
    g = rng_for(seed)
    return g.integers(1, cols + 1, size=rows, dtype=np.int64).astype(np.int32)


# --------------------------------------------------------------------------
# Named workloads
# --------------------------------------------------------------------------

WORKLOADS = (
    "sampling_f32_4x8192_k64",
    "indexer_bf16_4096x2048_causal_k512_gather",
    "indexer_bf16_4x204800_k1024",
    "sampling_f32_256x131072_k4096_nan",
    "indexer_bf16_3x4096x16384_levels64_k2048_gather",
)

DESCRIPTIONS = {
    "sampling_f32_4x8192_k64":
        "fp32 top-k: x[4, 8192] N(0,1), k=64, all columns valid, sorted indices, int32, values",
    "indexer_bf16_4096x2048_causal_k512_gather":
        "bf16 indexer top-k: scores[4096, 2048] N(0,1), row_end[i]=min(2048, i//2+1), k=512, "
        "unsorted int32, no values; then gather of the 512 selected rows from key[1, 2048, 128] bf16",
    "indexer_bf16_4x204800_k1024":
        "bf16 top-k: x[4, 204800] N(0,1), k=1024, sorted int32 indices, values",
    "sampling_f32_256x131072_k4096_nan":
        "fp32 sampling top-k: logits[256, 131072] = 2*N(0,1), +8 at 32 random columns per row, "
        "one NaN at a seeded (row, col), k=4096, sorted int64 indices, values",
    "indexer_bf16_3x4096x16384_levels64_k2048_gather":
        "bf16 indexer top-k at batch 3: scores[12288, 16384] on 64 levels (heavy ties), "
        "row_end ~ U{1..16384}, k=2048, unsorted int32; then gather of 512 positions per row "
        "from key[3, 16384, 128] bf16 with batch offset b*16384",
}


def workload(name: str, rows: int | None = None) -> dict:
    """Build one named workload.

    ``rows`` (optional) keeps only the first ``rows`` score rows (same seed, so
    row i is the same row as in the full workload; the key is kept whole).
    Returns a dict with the fields the top-k / gather calls take:
    ``x`` (bit array [R, stride]), ``dtype``, ``rows``, ``cols``, ``stride``,
    ``row_end`` (int32 [R] or None), ``k``, ``sorted_index``, ``idx_dtype``,
    ``want_values`` and, for gather workloads, ``key`` (bf16 bits
    [b, comp_len, d]), ``b``, ``comp_len``, ``d``, ``n_gather``,
    ``rows_per_batch``, plus ``nan_at`` (row, col) where a NaN was planted.
    """
    if name not in WORKLOADS:
        raise KeyError(name)
    seed = SEED_BASE + 1 + WORKLOADS.index(name)
    w: dict = {"name": name, "description": DESCRIPTIONS[name], "nan_at": None, "key": None}
    if name == "sampling_f32_4x8192_k64":
        R, C = 4, 8192
        x = normal_rows(seed, R, C, F32)
        w.update(dtype=F32, cols=C, stride=C, row_end=None, k=64, sorted_index=True,
                 idx_dtype=I32, want_values=True)
    elif name == "indexer_bf16_4096x2048_causal_k512_gather":
        R, C = 4096, 2048
        x = normal_rows(seed, R, C, BF16)
        key = f32_to_bf16_bits(rng_for(seed + 100).standard_normal((1, 2048, 128), dtype=np.float32))
        w.update(dtype=BF16, cols=C, stride=C, row_end=causal_row_end(R, C), k=512,
                 sorted_index=False, idx_dtype=I32, want_values=False,
                 key=key, b=1, comp_len=2048, d=128, n_gather=512)
    elif name == "indexer_bf16_4x204800_k1024":
        R, C = 4, 204800
        # 204800 bf16 = 409600 B = 3200 x 128 B: the row stride is already a 128-byte multiple.
        x = normal_rows(seed, R, C, BF16)
        w.update(dtype=BF16, cols=C, stride=C, row_end=None, k=1024, sorted_index=True,
                 idx_dtype=I32, want_values=True)
    elif name == "sampling_f32_256x131072_k4096_nan":
        R, C = 256, 131072
        g = rng_for(seed)
        v = g.standard_normal((R, C), dtype=np.float32) * np.float32(2.0)
        for r in range(R):
            cols = g.choice(C, size=32, replace=False)
            v[r, cols] += np.float32(8.0)
        nr = int(g.integers(0, R))
        nc = int(g.integers(0, C))
        v[nr, nc] = np.float32(np.nan)
        x = f32_to_bits(v)
        w.update(dtype=F32, cols=C, stride=C, row_end=None, k=4096, sorted_index=True,
                 idx_dtype=I64, want_values=True, nan_at=(nr, nc))
    else:  # indexer_bf16_3x4096x16384_levels64_k2048_gather
        B, Rb, C = 3, 4096, 16384
        R = B * Rb
        x = levels64_bf16(seed, R, C)
        key = f32_to_bf16_bits(rng_for(seed + 100).standard_normal((B, C, 128), dtype=np.float32))
        w.update(dtype=BF16, cols=C, stride=C, row_end=uniform_row_end(seed + 200, R, C), k=2048,
                 sorted_index=False, idx_dtype=I32, want_values=False,
                 key=key, b=B, comp_len=C, d=128, n_gather=512)
    w["x"] = x
    w["rows"] = x.shape[0]
    if rows is not None and rows < w["rows"]:
        w["x"] = x[:rows].copy()
        if w["row_end"] is not None:
            w["row_end"] = w["row_end"][:rows].copy()
        w["rows"] = rows
        if w["nan_at"] is not None and w["nan_at"][0] >= rows:
            w["nan_at"] = None
    if w["key"] is not None:
        w["rows_per_batch"] = x.shape[0] // w["b"]
    return w


def row_subset(w: dict, row_ids) -> dict:
    """A copy of workload ``w`` restricted to the given rows (for the oracle on samples)."""
    row_ids = np.asarray(row_ids, dtype=np.int64)
    s = dict(w)
    s["x"] = np.ascontiguousarray(w["x"][row_ids])
    s["row_end"] = None if w["row_end"] is None else np.ascontiguousarray(w["row_end"][row_ids])
    s["rows"] = len(row_ids)
    s["row_ids"] = row_ids
    return s


def gather_positions(seed: int, rows: int, n: int, comp_len: int, neg_frac: float = 0.0) -> np.ndarray:
    """Seeded int32 positions [rows, n] in [0, comp_len), a fraction set to -1."""
    g = rng_for(seed)
    pos = g.integers(0, comp_len, size=(rows, n), dtype=np.int64)
    if neg_frac > 0:
        pos[g.random((rows, n)) < neg_frac] = -1
    return pos.astype(np.int32)


def kl_pair_gather(rows: int = 1024, n: int = 512, comp_len: int = 2048, d: int = 128, d2: int = 512, b: int = 1,
                   seed: int = SEED_BASE + 6) -> dict:
    """Inputs of the Indexer KL loss's double gather.

    MindSpore hyper-parallel pull request "perf/gather-index-select": per
    query chunk the loss gathers 1024 rows x 512 selected positions twice,
    from the index key (head_dim 128) and from the attention key (512), at
    compressed length 2048.  Keys are bf16 N(0,1) [b, comp_len, d|d2];
    positions are uniform in [0, comp_len) with 2% set to -1 (the fills of
    short rows, read as position 0).
    """
    g = rng_for(seed)
    key = f32_to_bf16_bits(g.standard_normal((b, comp_len, d), dtype=np.float32))
    key2 = f32_to_bf16_bits(g.standard_normal((b, comp_len, d2), dtype=np.float32))
    pos = gather_positions(seed + 1, rows, n, comp_len, neg_frac=0.02)
    return {"key": key, "key2": key2, "pos": pos, "rows": rows, "n": n, "comp_len": comp_len, "d": d, "d2": d2,
            "b": b}


def block_candidates_workload(rows: int = 1024, comp_len: int = 2048, block_size: int = 64, topk_blocks: int = 16,
                              d: int = 128, seed: int = SEED_BASE + 7) -> dict:
    """Inputs of the block-level candidate chain (MindSpore hyper-parallel pull request
    "perf/gather-index-select": per query chunk of 1024 rows the chain gathers
    topk_blocks * block_size = 1024 positions at compressed length 2048, head_dim 128).

    Block scores bf16 N(0,1) [rows, comp_len / block_size]; causal position ends
    pos_end[i] = min(comp_len, 2 (i + 1)) (the chunk's rows spread over the compressed
    length, so early rows hold fewer candidate blocks than topk_blocks); key bf16 N(0,1)
    [1, comp_len, d].
    """
    g = rng_for(seed)
    n_blocks = comp_len // block_size
    scores = f32_to_bf16_bits(g.standard_normal((rows, n_blocks), dtype=np.float32))
    key = f32_to_bf16_bits(g.standard_normal((1, comp_len, d), dtype=np.float32))
    pos_end = np.minimum(comp_len, 2 * (np.arange(rows) + 1)).astype(np.int32)
    return {"scores": scores, "key": key, "pos_end": pos_end, "rows": rows, "n_blocks": n_blocks,
            "block_size": block_size, "topk_blocks": topk_blocks, "comp_len": comp_len, "d": d}
