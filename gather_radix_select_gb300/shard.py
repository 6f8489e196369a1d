"""Rows of one top-k (+ gather) call sharded over several GPUs, one process per GPU.

Rows are independent, so the work splits by rows with no exchange on the data
path; each rank selects (and gathers) its own rows and the outputs are put
back in row order.  How the rows are cut follows the PaddleFleet pull request
"Balance the latent-MQA indexer's CP rows with a dual-chunk swap"
(description): with causal row ends, row i has about i valid columns, so
contiguous row blocks would hand the last rank most of the work; cutting the
rows into 2 * world chunks and giving rank g chunks g and 2 * world - 1 - g
gives every rank about the same number of valid columns.

Nothing here computes a selection: ``run_rank`` calls a compute function for
each of a rank's row pieces (the library call, see ``topk_pieces``), and
``assemble`` puts the pieces of all ranks back in row order.  The pieces are
cut at batch boundaries, so a fused gather sees one key batch per piece and
the batch offset (batch = row / rows_per_batch) stays the global one.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def _cuts(n: int, parts: int) -> list[int]:
    """Boundaries of `parts` contiguous pieces of [0, n) whose sizes differ by at most one."""
    return [n * i // parts for i in range(parts + 1)]


def partition_rows(rows: int, world: int, mode: str = "blocks") -> list[list[tuple[int, int]]]:
    """Row ranges [start, stop) of every rank, in row order.

    "blocks": one contiguous block per rank (sizes differ by at most one), for rows of equal width.
    "dual_chunk": the rows cut into 2 * world chunks; rank g takes chunks g and 2 * world - 1 - g,
    for row ends that grow (or shrink) along the batch, such as causal masks."""
    if rows < 0 or world < 1:
        raise ValueError("rows must be >= 0 and world >= 1")
    if mode == "blocks":
        c = _cuts(rows, world)
        return [[(c[g], c[g + 1])] if c[g] < c[g + 1] else [] for g in range(world)]
    if mode == "dual_chunk":
        c = _cuts(rows, 2 * world)
        out = []
        for g in range(world):
            rs = [r for r in [(c[g], c[g + 1]), (c[2 * world - 1 - g], c[2 * world - g])] if r[0] < r[1]]
            if len(rs) == 2 and rs[0][1] == rs[1][0]:  # the middle rank's two chunks touch
                rs = [(rs[0][0], rs[1][1])]
            out.append(rs)
        return out
    raise ValueError("mode must be 'blocks' or 'dual_chunk'")


def split_at_batches(ranges: list[tuple[int, int]], rows_per_batch: int) -> list[tuple[int, int, int]]:
    """(start, stop, batch) pieces of the ranges, each inside one batch of rows_per_batch rows."""
    if rows_per_batch < 1:
        raise ValueError("rows_per_batch must be >= 1")
    out = []
    for s, e in ranges:
        while s < e:
            b = s // rows_per_batch
            t = min(e, (b + 1) * rows_per_batch)
            out.append((s, t, b))
            s = t
    return out


def call_pieces(ranges: list[tuple[int, int]], rows_per_batch: int) -> list[tuple[int, int, int, int]]:
    """(start, stop, first_batch, stop_batch) pieces of the ranges that one fused call can take: either
    whole consecutive batches (start and stop on batch boundaries; the call sees key batches
    [first_batch, stop_batch)) or a part of one batch (stop_batch = first_batch + 1)."""
    out = []
    for s, e, b in split_at_batches(ranges, rows_per_batch):
        whole = s == b * rows_per_batch and e == (b + 1) * rows_per_batch
        if whole and out:
            ps, pe, pb0, pb1 = out[-1]
            if pe == s and ps == pb0 * rows_per_batch and pe == pb1 * rows_per_batch:  # extends whole batches
                out[-1] = (ps, e, pb0, b + 1)
                continue
        out.append((s, e, b, b + 1))
    return out


@dataclass
class Piece:
    """Outputs of one row piece [start, stop) of one rank."""
    start: int
    stop: int
    values: object = None   # [stop - start, k] or None
    indices: object = None  # [stop - start, k]
    gathered: object = None  # [stop - start, n_gather, d] or None


def run_rank(compute, ranges: list[tuple[int, int]], rows_per_batch: int | None = None) -> list[Piece]:
    """One rank's share: compute(start, stop, batches) -> (values, indices, gathered) for every piece of
    its ranges.  With rows_per_batch the pieces are those of call_pieces and batches = (first, stop)
    key batches; without, the ranges as they are and batches = None."""
    pieces = call_pieces(ranges, rows_per_batch) if rows_per_batch else [(s, e, None, None) for s, e in ranges]
    out = []
    for s, e, b0, b1 in pieces:
        v, i, gth = compute(s, e, None if b0 is None else (b0, b1))
        out.append(Piece(s, e, v, i, gth))
    return out


def assemble(pieces: list[Piece], rows: int, cat):
    """(values, indices, gathered) in row order from the pieces of every rank; `cat` concatenates a
    list of arrays or tensors along rows (np.concatenate, torch.cat).  Every row must be covered
    exactly once."""
    pieces = sorted(pieces, key=lambda p: p.start)
    at = 0
    for p in pieces:
        if p.start != at:
            raise ValueError("pieces do not cover the rows exactly once (gap or overlap at row %d)" % at)
        at = p.stop
    if at != rows:
        raise ValueError("pieces cover %d of %d rows" % (at, rows))

    def join(field):
        parts = [getattr(p, field) for p in pieces]
        if any(x is None for x in parts):
            return None
        return cat(parts) if parts else None

    return join("values"), join("indices"), join("gathered")


def rows_of(ranges: list[tuple[int, int]]) -> np.ndarray:
    """The global row ids of a rank's ranges, in order."""
    if not ranges:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([np.arange(s, e, dtype=np.int64) for s, e in ranges])


def topk_pieces(x, k: int, *, end=None, key=None, n_gather: int = 0, **topk_args):
    """compute() for run_rank through this library: the top-k (and, with a key, the fused gather) of
    rows [start, stop) of x (and end), reading key batches [first, stop) of key (a [b, comp_len, d]
    tensor).  Rows of several pieces go to separate calls; nothing is copied."""
    import gather_radix_select_gb300 as g

    def compute(s, e, batches):
        xs = x[s:e]
        es = None if end is None else end[s:e]
        if key is not None and n_gather > 0:
            kb = key[batches[0]:batches[1]] if batches is not None else key
            v, i, gth = g.topk_gather(xs, k, kb, n_gather, end=es, **topk_args)
            return v, i, gth
        v, i = g.topk(xs, k, end=es, **topk_args)
        return v, i, None

    return compute
