"""ctypes binding of libsel.so (include/sel.h).  Argument marshalling only.

The library is built in-tree by ``gather_radix_select_gb300.build``; loading
fails loudly (``RuntimeError``) when it is missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SEL_OK, SEL_EINVAL, SEL_EALIGN, SEL_EUNSUPPORTED, SEL_ECUDA, SEL_ETIMEOUT, SEL_ESCRATCH, SEL_EBOUNDS = range(8)
SEL_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
SEL_F32, SEL_BF16 = 0, 1
SEL_I32, SEL_I64 = 0, 1
SEL_MAX_K = 4096
# include/sel_tuning.h
SEL_TUNE_PLAN, SEL_TUNE_PARTS, SEL_TUNE_ROW_SAMPLE, SEL_TUNE_HIST_AGG, SEL_TUNE_ROW_ORDER = range(5)
SEL_PLANS = {"auto": -1, "reg": 0, "row": 1, "wide": 2, "split": 3, "stream": 4, "flat": 5}

# every symbol include/sel.h declares, with its ctypes signature
_vp, _i64, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
SIGNATURES = {
    "sel_stride_requirement": (_int, [ctypes.POINTER(_int), ctypes.POINTER(_int)]),
    "sel_topk": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _int, _int, _int, _int,
                        _vp, _i64, _vp, _i64, _vp, ctypes.c_size_t, _vp, _vp, _vp]),
    "sel_topk_workspace_size": (ctypes.c_size_t, [_int, _i64, _i64, _int]),
    "sel_max_cols": (_i64, [_int]),
    "sel_gather_rows": (_int, [_vp, _i64, _i64, _i64, _i64, _i64, _vp, _int, _i64, _i64, _i64,
                               _vp, _vp, _vp]),
    "sel_gather_rows_pair": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _i64, _i64, _i64, _vp, _int,
                                    _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "sel_block_topk_gather": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _int, _i64, _vp, _i64,
                                     _vp, _i64, _i64, _i64, _i64, _i64, _vp,
                                     _vp, ctypes.c_size_t, _vp, _vp, _vp]),
    "sel_topk_gather": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _int, _int, _int, _int,
                               _vp, _i64, _vp, _i64,
                               _vp, _i64, _i64, _i64, _i64, _i64, _i64, _vp,
                               _vp, ctypes.c_size_t, _vp, _vp, _vp]),
    "sel_topk_noalloc": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _int, _int, _int, _int,
                                _vp, _i64, _vp, _i64, _vp, _vp, _vp]),
    "sel_strerror": (ctypes.c_char_p, [_int]),
    "sel_topk_kernel_name": (ctypes.c_char_p, [_int, _i64, _i64, _int, _i64]),
    "sel_set_tuning": (_int, [_int, _int]),
    "sel_get_tuning": (_int, [_int]),
    "sel_selftest_wait_timeout": (_int, [_vp, ctypes.c_longlong, _vp]),
    "sel_debug_build": (_int, []),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """libsel.so, or the bounds-checked libsel_debug.so when SEL_LIBRARY=debug is set (read when the
    library is first loaded)."""
    return _build.DEBUG_SO if os.environ.get("SEL_LIBRARY", "") == "debug" else _build.SO


def load(build_if_missing: bool = False):
    """Load libsel.so once.  Raises RuntimeError when it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    "libsel.so is not built (%s); run `python -m gather_radix_select_gb300.build`" % path)
            _build.build(debug=path == _build.DEBUG_SO)
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class SelError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().sel_strerror(status).decode()
        super().__init__("%s failed: %s (status %d)" % (where, msg, status))
        self.status = status


def check(status: int, where: str) -> None:
    if status != SEL_OK:
        raise SelError(status, where)
