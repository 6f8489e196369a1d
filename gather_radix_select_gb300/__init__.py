"""gather_radix_select_gb300 -- batched row-wise top-k and flat row gather on GB300.

Python face of the C ABI in ``include/sel.h`` (libsel.so, built in-tree for
sm_103a by ``gather_radix_select_gb300.build``).  PyTorch supplies device
memory and the current CUDA stream; every step of the computation runs in
the library's kernels.  There is no CPU fallback: without the built library
every call raises ``RuntimeError``.

API shape after "Speed up PyTorch TopK with DeepSelect" ("Basic TopK usage",
"Returning indices only", "Handling stride alignment", "Using an existing
index buffer", "Working with variable-length rows") and, for the gather,
the MindSpore hyper-parallel pull request "perf/gather-index-select".
"""
from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import SelError, SEL_MAX_K

__all__ = ["topk", "gather_rows", "gather_rows_pair", "topk_gather", "block_topk_gather", "stride_requirement", "max_cols", "workspace_size", "kernel_name",
           "set_tuning", "get_tuning", "SelError",
           "SEL_MAX_K", "library_path"]

_DTYPES = {torch.float32: _native.SEL_F32, torch.bfloat16: _native.SEL_BF16}
_IDX = {torch.int32: _native.SEL_I32, torch.int64: _native.SEL_I64}


def library_path() -> str:
    return _native.library_path()


_ALIGN = None


def stride_requirement() -> tuple[int, int]:
    """(input_alignment, output_alignment) in bytes, as in ``get_stride_requirement()``."""
    global _ALIGN
    if _ALIGN is None:
        a, b = ctypes.c_int(), ctypes.c_int()
        _native.check(_native.load().sel_stride_requirement(ctypes.byref(a), ctypes.byref(b)),
                      "sel_stride_requirement")
        _ALIGN = (a.value, b.value)
    return _ALIGN


def max_cols(dtype: torch.dtype = torch.float32) -> int:
    """Widest row ``topk`` accepts for ``dtype`` on the current device."""
    return int(_native.load().sel_max_cols(_DTYPES[dtype]))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


_WORKSPACES: dict = {}


def workspace_size(dtype: torch.dtype, rows: int, cols: int, k: int, device=None) -> int:
    """Scratch bytes a top-k call of this shape needs on ``device`` (0 for most shapes)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(_native.load().sel_topk_workspace_size(_DTYPES[dtype], rows, cols, int(k)))


def kernel_name(dtype: torch.dtype, rows: int, cols: int, k: int, n_gather: int = 0, device=None) -> str:
    """Kernel a top-k (n_gather == 0) or fused top-k + gather call of this shape launches on ``device``."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        name = _native.load().sel_topk_kernel_name(_DTYPES[dtype], rows, cols, int(k), int(n_gather))
    if name is None:
        raise ValueError("invalid shape for kernel_name")
    return name.decode()


_KNOBS = {"plan": _native.SEL_TUNE_PLAN, "parts": _native.SEL_TUNE_PARTS,
          "row_sample": _native.SEL_TUNE_ROW_SAMPLE, "hist_agg": _native.SEL_TUNE_HIST_AGG,
          "row_order": _native.SEL_TUNE_ROW_ORDER}


def set_tuning(plan: str | None = None, parts: int | None = None, row_sample: bool | None = None,
               hist_agg: bool | None = None, row_order: bool | None = None) -> None:
    """Tuning and test hooks (include/sel_tuning.h); None leaves a knob as it is.

    ``plan``: "auto" or the kernel to force where it can run a shape ("reg", "row", "wide",
    "split", "stream", "flat").  ``parts``: parts per row of the streaming kernel's split mode
    (0 = automatic).  ``row_order``: with per-row ends, CTAs take rows from both ends of the batch
    alternately (default False: in order, measured faster).  Process-wide; takes effect on the next call."""
    lib = _native.load()
    vals = {"plan": None if plan is None else _native.SEL_PLANS[plan], "parts": parts,
            "row_sample": None if row_sample is None else int(bool(row_sample)),
            "hist_agg": None if hist_agg is None else int(bool(hist_agg)),
            "row_order": None if row_order is None else int(bool(row_order))}
    for name, v in vals.items():
        if v is not None:
            _native.check(lib.sel_set_tuning(_KNOBS[name], int(v)), "sel_set_tuning(%s)" % name)


def get_tuning() -> dict:
    """The knobs' current values, in the form set_tuning takes."""
    lib = _native.load()
    plans = {v: k for k, v in _native.SEL_PLANS.items()}
    return {"plan": plans[lib.sel_get_tuning(_native.SEL_TUNE_PLAN)],
            "parts": int(lib.sel_get_tuning(_native.SEL_TUNE_PARTS)),
            "row_sample": bool(lib.sel_get_tuning(_native.SEL_TUNE_ROW_SAMPLE)),
            "hist_agg": bool(lib.sel_get_tuning(_native.SEL_TUNE_HIST_AGG)),
            "row_order": bool(lib.sel_get_tuning(_native.SEL_TUNE_ROW_ORDER))}


def _workspace(nbytes: int, device, stream):
    """A scratch buffer of >= nbytes, cached per (device, stream) (calls on one stream never overlap)."""
    if nbytes == 0:
        return None, 0
    key = (device.index, stream.cuda_stream)
    buf = _WORKSPACES.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _WORKSPACES[key] = buf
    return buf, buf.numel()


def _padded_rows(rows: int, k: int, dtype: torch.dtype, device) -> torch.Tensor:
    """[rows, k] view of a buffer whose row stride is a multiple of the output alignment."""
    _, out_align = stride_requirement()
    es = torch.empty((), dtype=dtype).element_size()
    per = max(1, out_align // es)
    stride = (k + per - 1) // per * per
    return torch.empty((rows, stride), dtype=dtype, device=device)[:, :k]


def _check_x(x: torch.Tensor):
    if x.dim() != 2:
        raise ValueError("x must be 2-D (batch_size, vocab_size)")
    if x.dtype not in _DTYPES:
        raise TypeError("x must be torch.float32 or torch.bfloat16")
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if x.size(1) > 1 and x.stride(1) != 1:
        raise ValueError("the last dimension of x must be contiguous")


def _check_end(end, rows, device):
    if end is None:
        return None
    if end.dtype != torch.int32 or end.dim() != 1 or end.numel() != rows or not end.is_cuda or not end.is_contiguous():
        raise ValueError("end must be a contiguous int32 CUDA tensor with one entry per row")
    if end.device != device:
        raise ValueError("end must be on x's device")
    return end


def _out_idx(output_idx, rows, k, indices_type, dev):
    """The caller's [rows, >=k] index buffer, checked, or a new padded one."""
    if indices_type not in _IDX:
        raise TypeError("indices_type must be torch.int32 or torch.int64")
    if output_idx is None:
        return _padded_rows(rows, k, indices_type, dev)
    if output_idx.dtype != indices_type or output_idx.dim() != 2 or output_idx.shape[0] != rows \
            or output_idx.shape[1] < k or (rows > 1 and output_idx.stride(1) != 1) or output_idx.device != dev:
        raise ValueError("output_idx must be a [rows, >=k] %s tensor on x's device" % indices_type)
    return output_idx


def _out_val(output_val, rows, k, dtype, dev):
    """The caller's [rows, >=k] value buffer, checked, or a new padded one."""
    if output_val is None:
        return _padded_rows(rows, k, dtype, dev)
    if output_val.dtype != dtype or output_val.dim() != 2 or output_val.shape[0] != rows \
            or output_val.shape[1] < k or (rows > 1 and output_val.stride(1) != 1) or output_val.device != dev:
        raise ValueError("output_val must be a [rows, >=k] tensor of x's dtype on x's device")
    return output_val


def _row_stride(x):
    return x.stride(0) if x.size(0) > 1 else max(x.stride(0), x.size(1))


def _order(sorted_index: bool, sorted_value: bool) -> int:
    # SEL_UNSORTED / SEL_SORT_INDEX / SEL_SORT_VALUE
    if sorted_index and sorted_value:
        raise ValueError("sorted_index and sorted_value exclude each other")
    return 2 if sorted_value else int(bool(sorted_index))


def topk(x: torch.Tensor, k: int, *, end: torch.Tensor | None = None, sorted_index: bool = False,
         sorted_value: bool = False, indices_type: torch.dtype = torch.int32, return_value: bool = True,
         output_idx: torch.Tensor | None = None, output_val: torch.Tensor | None = None,
         nan_flag: torch.Tensor | None = None, err_flag: torch.Tensor | None = None, stream=None,
         workspace: torch.Tensor | None = None):
    """Row-wise top-k of a 2-D CUDA tensor (largest values; ties: smaller index).

    Returns ``(values, indices)``; ``values`` is None when ``return_value``
    is False.  Rows shorter than k (per ``end``) are filled with index -1 and
    value -inf.  ``sorted_index``: each row by index ascending;
    ``sorted_value``: by value descending, equal values by index (ranked in the
    selection launch when the plan is the staged row kernel, else a second
    launch).  Outputs may be non-contiguous (row strides padded to the
    output alignment).  ``nan_flag`` / ``err_flag`` are optional caller-zeroed
    int32 CUDA tensors the kernel ORs / writes into.  ``output_idx`` /
    ``output_val`` are optional caller-owned [rows, >=k] buffers (row strides
    a multiple of the output alignment); results go to their first k columns.
    ``workspace`` (uint8 CUDA tensor) is only needed when few wide rows are
    split over several CTAs; by default a cached buffer is used.
    """
    _check_x(x)
    order = _order(sorted_index, sorted_value)
    rows, cols = x.shape
    dev = x.device
    end = _check_end(end, rows, dev)
    idx = _out_idx(output_idx, rows, k, indices_type, dev)
    val = _out_val(output_val, rows, k, x.dtype, dev) if return_value else None
    with torch.cuda.device(dev):
        lib = _native.load()
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        ws, ws_bytes = _ws_for(lib, workspace, x.dtype, rows, cols, k, dev, s)
        st = lib.sel_topk(
            _ptr(x), _DTYPES[x.dtype], rows, cols, _row_stride(x), _ptr(end), int(k), order,
            _IDX[indices_type], int(bool(return_value)), _ptr(idx), idx.stride(0) if rows > 1 else max(idx.stride(0), k),
            _ptr(val), 0 if val is None else (val.stride(0) if rows > 1 else max(val.stride(0), k)),
            _ptr(ws), ws_bytes, _ptr(nan_flag), _ptr(err_flag), ctypes.c_void_p(s.cuda_stream))
    _native.check(st, "sel_topk")
    if output_val is not None and val is not None:
        val = val[:, :k]
    return val, idx[:, :k] if output_idx is not None else idx


def _ws_for(lib, workspace, dtype, rows, cols, k, dev, s):
    need = int(lib.sel_topk_workspace_size(_DTYPES[dtype], rows, cols, int(k))) if rows > 0 else 0
    if workspace is not None:
        if workspace.dtype != torch.uint8 or not workspace.is_cuda or workspace.numel() < need:
            raise ValueError("workspace must be a uint8 CUDA tensor of at least %d bytes" % need)
        return workspace, workspace.numel()
    return _workspace(need, dev, s)


def _key_strides(key):
    if key.dim() != 3 or key.dtype != torch.bfloat16 or not key.is_cuda:
        raise ValueError("key must be a 3-D bf16 CUDA tensor [b, comp_len, d]")
    if key.size(2) > 1 and key.stride(2) != 1:
        raise ValueError("key rows must be contiguous in their last dimension")
    return key.stride(0), key.stride(1)


def gather_rows(key: torch.Tensor, idx: torch.Tensor, *, out: torch.Tensor | None = None,
                err_flag: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[r, j, :] = key[r // (rows // b), max(idx[r, j], 0), :] as one flat-index gather.

    key: bf16 [b, comp_len, d] (rows may be strided); idx: int32/int64 [rows, n]
    with rows a multiple of b.  A position >= comp_len yields a zero row and
    sets ``err_flag``.
    """
    kbs, krs = _key_strides(key)
    b, comp_len, d = key.shape
    if idx.dim() != 2 or idx.dtype not in _IDX or idx.device != key.device:
        raise ValueError("idx must be a 2-D int32/int64 tensor on key's device")
    if idx.size(1) > 1 and idx.stride(1) != 1:
        raise ValueError("idx rows must be contiguous")
    rows, n = idx.shape
    if out is None:
        out = torch.empty((rows, n, d), dtype=torch.bfloat16, device=key.device)
    elif out.shape != (rows, n, d) or not out.is_contiguous() or out.dtype != torch.bfloat16 \
            or out.device != key.device:
        raise ValueError("out must be a contiguous bf16 [rows, n, d] tensor")
    with torch.cuda.device(key.device):
        st = _native.load().sel_gather_rows(
            _ptr(key), b, comp_len, d, kbs, krs, _ptr(idx), _IDX[idx.dtype], rows, n,
            idx.stride(0) if rows > 1 else max(idx.stride(0), n), _ptr(out), _ptr(err_flag),
            _stream(key.device, stream))
    _native.check(st, "sel_gather_rows")
    return out


def gather_rows_pair(key: torch.Tensor, key2: torch.Tensor, idx: torch.Tensor, *, out: torch.Tensor | None = None,
                     out2: torch.Tensor | None = None, err_flag: torch.Tensor | None = None, stream=None):
    """``gather_rows`` of two keys at the same positions, in one launch.

    key: bf16 [b, comp_len, d]; key2: bf16 [b, comp_len, d2] (same b and
    comp_len, each may be strided); idx: int32/int64 [rows, n].  Returns
    ``(out, out2)``, bf16 [rows, n, d] and [rows, n, d2].
    """
    kbs, krs = _key_strides(key)
    kbs2, krs2 = _key_strides(key2)
    b, comp_len, d = key.shape
    if key2.shape[0] != b or key2.shape[1] != comp_len or key2.device != key.device:
        raise ValueError("key2 must be [b, comp_len, d2] with key's b and comp_len, on key's device")
    d2 = key2.shape[2]
    if idx.dim() != 2 or idx.dtype not in _IDX or idx.device != key.device:
        raise ValueError("idx must be a 2-D int32/int64 tensor on key's device")
    if idx.size(1) > 1 and idx.stride(1) != 1:
        raise ValueError("idx rows must be contiguous")
    rows, n = idx.shape
    outs = []
    for o, dd in ((out, d), (out2, d2)):
        if o is None:
            o = torch.empty((rows, n, dd), dtype=torch.bfloat16, device=key.device)
        elif o.shape != (rows, n, dd) or not o.is_contiguous() or o.dtype != torch.bfloat16 \
                or o.device != key.device:
            raise ValueError("outputs must be contiguous bf16 [rows, n, d] tensors")
        outs.append(o)
    with torch.cuda.device(key.device):
        st = _native.load().sel_gather_rows_pair(
            _ptr(key), d, kbs, krs, _ptr(key2), d2, kbs2, krs2, b, comp_len, _ptr(idx), _IDX[idx.dtype], rows, n,
            idx.stride(0) if rows > 1 else max(idx.stride(0), n), _ptr(outs[0]), _ptr(outs[1]), _ptr(err_flag),
            _stream(key.device, stream))
    _native.check(st, "sel_gather_rows_pair")
    return outs[0], outs[1]


def block_topk_gather(scores: torch.Tensor, topk_blocks: int, block_size: int, *,
                      pos_end: torch.Tensor | None = None, key: torch.Tensor | None = None,
                      out_pos: torch.Tensor | None = None, gather_out: torch.Tensor | None = None,
                      nan_flag: torch.Tensor | None = None, err_flag: torch.Tensor | None = None, stream=None,
                      workspace: torch.Tensor | None = None):
    """Block-level candidate selection: the ``topk_blocks`` best blocks of each row of
    ``scores`` [rows, n_blocks] (blocks of ``block_size`` positions; a block is a candidate
    when it holds a position below ``pos_end[r]``), expanded to their valid positions in
    ascending order then -1 (int32 [rows, topk_blocks * block_size]), and, with ``key``
    (bf16 [b, comp_len, d]), the key rows gathered there.  Returns ``(positions, gathered)``,
    ``gathered`` None without ``key``.
    """
    _check_x(scores)
    rows, n_blocks = scores.shape
    dev = scores.device
    pos_end = _check_end(pos_end, rows, dev)
    npos = int(topk_blocks) * int(block_size)
    if out_pos is None:
        pos = _padded_rows(rows, npos, torch.int32, dev)
    else:
        pos = out_pos
        if pos.dtype != torch.int32 or pos.dim() != 2 or pos.shape[0] != rows or pos.shape[1] < npos \
                or (rows > 1 and pos.stride(1) != 1) or pos.device != dev:
            raise ValueError("out_pos must be an int32 [rows, >=topk_blocks*block_size] tensor on scores' device")
    b = comp_len = d = kbs = krs = 0
    if key is not None:
        kbs, krs = _key_strides(key)
        b, comp_len, d = key.shape
        if key.device != dev:
            raise ValueError("key must be on scores' device")
        if gather_out is None:
            gather_out = torch.empty((rows, npos, d), dtype=torch.bfloat16, device=dev)
        elif gather_out.shape != (rows, npos, d) or not gather_out.is_contiguous() \
                or gather_out.dtype != torch.bfloat16 or gather_out.device != dev:
            raise ValueError("gather_out must be a contiguous bf16 [rows, topk_blocks*block_size, d] tensor")
    else:
        gather_out = None
    with torch.cuda.device(dev):
        lib = _native.load()
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        ws, ws_bytes = _ws_for(lib, workspace, scores.dtype, rows, n_blocks, topk_blocks, dev, s)
        st = lib.sel_block_topk_gather(
            _ptr(scores), _DTYPES[scores.dtype], rows, n_blocks, _row_stride(scores), _ptr(pos_end),
            int(topk_blocks), int(block_size), _ptr(pos), pos.stride(0) if rows > 1 else max(pos.stride(0), npos),
            _ptr(key), b, comp_len, d, kbs, krs, _ptr(gather_out),
            _ptr(ws), ws_bytes, _ptr(nan_flag), _ptr(err_flag), ctypes.c_void_p(s.cuda_stream))
    _native.check(st, "sel_block_topk_gather")
    return (pos[:, :npos] if out_pos is not None else pos), gather_out


def topk_gather(x: torch.Tensor, k: int, key: torch.Tensor, n_gather: int, *, end: torch.Tensor | None = None,
                sorted_index: bool = False, sorted_value: bool = False, indices_type: torch.dtype = torch.int32,
                return_value: bool = False,
                return_indices: bool = True, gather_out: torch.Tensor | None = None,
                output_idx: torch.Tensor | None = None, output_val: torch.Tensor | None = None,
                nan_flag: torch.Tensor | None = None, err_flag: torch.Tensor | None = None, stream=None,
                workspace: torch.Tensor | None = None):
    """``topk`` then ``gather_rows`` of the first ``n_gather`` selected columns, in one launch.

    Returns ``(values, indices, gathered)`` with ``gathered`` bf16
    [rows, n_gather, d]; values / indices are None when not requested.  With
    ``sorted_value`` the gathered columns are the n_gather largest values, in
    value order (one launch when the plan is the staged row or register
    kernel, else the selection, then one launch that orders and gathers).
    """
    _check_x(x)
    order = _order(sorted_index, sorted_value)
    rows, cols = x.shape
    dev = x.device
    end = _check_end(end, rows, dev)
    kbs, krs = _key_strides(key)
    b, comp_len, d = key.shape
    if key.device != dev:
        raise ValueError("key must be on x's device")
    if not return_indices and order != 2:
        idx = None
    else:  # value order gathers from the ordered index rows, so they are always written
        idx = _out_idx(output_idx, rows, k, indices_type, dev)
    val = _out_val(output_val, rows, k, x.dtype, dev) if return_value else None
    if gather_out is None:
        gather_out = torch.empty((rows, n_gather, d), dtype=torch.bfloat16, device=dev)
    elif gather_out.shape != (rows, n_gather, d) or not gather_out.is_contiguous() \
            or gather_out.dtype != torch.bfloat16 or gather_out.device != dev:
        raise ValueError("gather_out must be a contiguous bf16 [rows, n_gather, d] tensor on x's device")
    with torch.cuda.device(dev):
        lib = _native.load()
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        ws, ws_bytes = _ws_for(lib, workspace, x.dtype, rows, cols, k, dev, s)
        st = lib.sel_topk_gather(
            _ptr(x), _DTYPES[x.dtype], rows, cols, _row_stride(x), _ptr(end), int(k), order,
            _IDX[indices_type], int(bool(return_value)),
            _ptr(idx), 0 if idx is None else (idx.stride(0) if rows > 1 else max(idx.stride(0), k)),
            _ptr(val), 0 if val is None else (val.stride(0) if rows > 1 else max(val.stride(0), k)),
            _ptr(key), b, comp_len, d, kbs, krs, int(n_gather), _ptr(gather_out),
            _ptr(ws), ws_bytes, _ptr(nan_flag), _ptr(err_flag), ctypes.c_void_p(s.cuda_stream))
    _native.check(st, "sel_topk_gather")
    if not return_indices:
        idx = None
    if idx is not None and output_idx is not None:
        idx = idx[:, :k]
    if val is not None and output_val is not None:
        val = val[:, :k]
    return val, idx, gather_out
