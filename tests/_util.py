"""Shared helpers for the tests: moving seeded bit arrays to torch and
checking top-k results against the oracle and against the definition."""
from __future__ import annotations

import numpy as np
import torch

import oracle

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}
IDX_DTYPE = {"i32": torch.int32, "i64": torch.int64}


def to_torch(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Bit array (uint32 fp32 / uint16 bf16) -> torch tensor of the float type on `device`."""
    if dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).view(torch.float32)
    else:
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def to_bits(t: torch.Tensor) -> np.ndarray:
    """Torch float tensor (any device) -> bit array (uint32 for fp32, uint16 for bf16)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


def valid_len(w, r):
    if w["row_end"] is None:
        return w["cols"]
    return int(min(max(int(w["row_end"][r]), 0), w["cols"]))


def compare_with_oracle(w, rows, gpu_idx, gpu_bits, sorted_index, skip_rows=()):
    """Exact comparison on the given rows: GPU output vs the oracle's.

    gpu_idx: int64 [len(rows), k]; gpu_bits: [len(rows), k] bit array or None.
    Unsorted output is compared as a set of (index, value bits) pairs; the
    fills must sit at the tail in both cases.
    """
    import synthetic as syn

    s = syn.row_subset(w, rows)
    o_idx, o_bits, o_nan = oracle.topk(s["x"], w["dtype"], w["k"], row_end=s["row_end"],
                                       sorted_index=sorted_index, cols=w["cols"])
    k = w["k"]
    checked = 0
    for i, r in enumerate(rows):
        if o_nan[i] or int(r) in skip_rows:
            continue
        n = valid_len(s, i)
        m = min(n, k)
        gi = np.asarray(gpu_idx[i], dtype=np.int64)
        assert (gi[m:] == -1).all(), "row %d: fills not at the tail" % r
        if sorted_index or n <= k:
            assert (gi[:m] == o_idx[i, :m]).all(), "row %d: indices differ" % r
            if gpu_bits is not None:
                assert (np.asarray(gpu_bits[i]).astype(np.uint32) == o_bits[i]).all(), "row %d: values differ" % r
        else:
            order_g = np.argsort(gi[:m], kind="stable")
            order_o = np.argsort(o_idx[i, :m], kind="stable")
            assert (gi[:m][order_g] == o_idx[i, :m][order_o]).all(), "row %d: index sets differ" % r
            if gpu_bits is not None:
                gb = np.asarray(gpu_bits[i]).astype(np.uint32)
                assert (gb[:m][order_g] == o_bits[i, :m][order_o]).all(), "row %d: values differ" % r
        if gpu_bits is not None and m < k:
            assert (np.asarray(gpu_bits[i][m:]).astype(np.uint32) == oracle.value_fill_bits(w["dtype"])).all()
        checked += 1
    return checked, o_nan


def check_definition_on_device(x: torch.Tensor, n_valid: torch.Tensor, k: int, idx: torch.Tensor,
                               vals: torch.Tensor | None, sorted_index: bool, skip_rows=(), chunk=256):
    """Property check of a whole top-k result, on the device, for every row.

    With t the smallest selected value of a row (n > k), the selection must be
    exactly {x > t} plus the first k - #{x > t} columns (in column order) with
    x == t, and the count must be k.  That characterises top-k with the
    smaller-index tie rule, so it proves the result at any size without the
    oracle.  Short rows (n <= k) must list 0..n-1 then -1.  Values must be the
    bits of x at the indices.
    """
    R, C = x.shape
    dev = x.device
    xf = x.float()
    cols = torch.arange(C, device=dev)
    skip = torch.zeros(R, dtype=torch.bool, device=dev)
    for r in skip_rows:
        skip[r] = True
    for r0 in range(0, R, chunk):
        r1 = min(R, r0 + chunk)
        xi = xf[r0:r1]
        nv = n_valid[r0:r1].to(torch.int64)
        ii = idx[r0:r1].to(torch.int64)
        sk = skip[r0:r1]
        pos = torch.arange(k, device=dev)[None, :]
        m = torch.minimum(nv, torch.tensor(k, device=dev))[:, None]
        valid_slot = pos < m
        # fills at the tail, in-range indices elsewhere
        assert bool(((ii == -1) | valid_slot).all()), "fill inside the valid part"
        assert bool(((ii >= 0) & (ii < nv[:, None]) | ~valid_slot).all()), "index out of range"
        short = nv <= k
        if bool(short.any()):
            exp = torch.where(valid_slot, pos.expand_as(ii), torch.full_like(ii, -1))
            bad = (ii != exp).any(dim=1) & short & ~sk
            assert not bool(bad.any()), "short row not 0..n-1"
        long_rows = ~short & ~sk
        if bool(long_rows.any()):
            li = ii[long_rows]
            lx = xi[long_rows]
            ln = nv[long_rows]
            inrow = cols[None, :] < ln[:, None]
            sel = torch.zeros_like(lx, dtype=torch.bool)
            sel.scatter_(1, li, True)
            assert bool((sel.sum(dim=1) == k).all()), "selected count != k (duplicates?)"
            selv = torch.gather(lx, 1, li)
            t = selv.min(dim=1).values[:, None]
            gt = (lx > t) & inrow
            eq = (lx == t) & inrow
            need = k - gt.sum(dim=1, keepdim=True)
            eq_rank = torch.cumsum(eq.to(torch.int64), dim=1)
            want = gt | (eq & (eq_rank <= need))
            assert bool((want == sel).all()), "selection differs from the definition"
            if sorted_index:
                assert bool((li[:, 1:] > li[:, :-1]).all()), "indices not ascending"
        if vals is not None:
            vi = vals[r0:r1]
            gidx = ii.clamp(min=0)
            xb = x[r0:r1]
            if x.dtype == torch.float32:
                xv = torch.gather(xb.view(torch.int32), 1, gidx)
                vv = vi.contiguous().view(torch.int32)
                fill = torch.tensor(0xFF800000 - (1 << 32), dtype=torch.int32, device=dev)
            else:
                xv = torch.gather(xb.view(torch.int16), 1, gidx)
                vv = vi.contiguous().view(torch.int16)
                fill = torch.tensor(0xFF80 - (1 << 16), dtype=torch.int16, device=dev)
            ok = torch.where(valid_slot, vv == xv, vv == fill)
            ok = ok | sk[:, None]
            assert bool(ok.all()), "values are not the bits of x at the indices"
