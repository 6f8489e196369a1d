"""The C-ABI library without a GPU: it builds, loads, exports every symbol
the headers under include/ declare, and rejects bad arguments on the host
before any CUDA call is made."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gather_radix_select_gb300 import _native
    return _native.load(build_if_missing=True)


def declared_symbols():
    names = set()
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(sel_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    assert declared_symbols() == sorted(["sel_block_topk_gather", "sel_gather_rows", "sel_gather_rows_pair",
                                         "sel_max_cols", "sel_stride_requirement",
                                         "sel_strerror", "sel_topk", "sel_topk_gather", "sel_topk_kernel_name",
                                         "sel_topk_noalloc", "sel_topk_workspace_size", "sel_set_tuning",
                                         "sel_get_tuning", "sel_selftest_wait_timeout", "sel_debug_build"])


def test_tuning_knobs_round_trip_and_reject_bad_values(lib):
    # host-only: the knobs are plain process state, no CUDA call is made
    import gather_radix_select_gb300 as g
    saved = g.get_tuning()
    try:
        for plan in ("reg", "row", "wide", "split", "stream", "flat", "auto"):
            g.set_tuning(plan=plan)
            assert g.get_tuning()["plan"] == plan
        g.set_tuning(parts=7, row_sample=True, hist_agg=True)
        g.set_tuning(row_order=False)
        assert g.get_tuning() == {"plan": "auto", "parts": 7, "row_sample": True, "hist_agg": True,
                                  "row_order": False}
        SEL_EINVAL = 1
        assert lib.sel_set_tuning(0, 99) == SEL_EINVAL   # no such plan
        assert lib.sel_set_tuning(0, -2) == SEL_EINVAL
        assert lib.sel_set_tuning(1, -1) == SEL_EINVAL   # negative parts
        assert lib.sel_set_tuning(42, 0) == SEL_EINVAL   # no such knob
        assert lib.sel_get_tuning(42) == -1
        assert g.get_tuning()["parts"] == 7              # a refused value changes nothing
    finally:
        g.set_tuning(**saved)


def test_wait_selftest_rejects_bad_arguments_on_the_host(lib):
    SEL_EINVAL = 1
    assert lib.sel_selftest_wait_timeout(None, 1000, None) == SEL_EINVAL
    flag = ctypes.c_int32(0)
    assert lib.sel_selftest_wait_timeout(ctypes.byref(flag), -1, None) == SEL_EINVAL


def test_every_declared_symbol_is_exported(lib):
    from gather_radix_select_gb300 import _native
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, name


def test_stride_requirement_and_messages(lib):
    a, b = ctypes.c_int(), ctypes.c_int()
    assert lib.sel_stride_requirement(ctypes.byref(a), ctypes.byref(b)) == 0
    assert (a.value, b.value) == (16, 16)
    assert lib.sel_stride_requirement(None, None) == 0
    for st in range(8):
        assert lib.sel_strerror(st) != b"unknown status"
    assert lib.sel_strerror(99) == b"unknown status"


FAKE = 0x10000  # never dereferenced: every call below is rejected on the host


def topk(lib, x=FAKE, dtype=0, rows=4, cols=64, stride=64, k=8, idx_dtype=0, want_values=0, out_idx=FAKE,
         out_idx_stride=8, out_val=None, out_val_stride=0, sorted_index=0):
    return lib.sel_topk(x, dtype, rows, cols, stride, None, k, sorted_index, idx_dtype, want_values, out_idx,
                        out_idx_stride, out_val, out_val_stride, None, 0, None, None, None)


def test_topk_rejections(lib):
    EINVAL, EALIGN = 1, 2
    assert topk(lib, k=0) == EINVAL
    assert topk(lib, k=4097) == EINVAL
    assert topk(lib, dtype=7) == EINVAL
    assert topk(lib, idx_dtype=3) == EINVAL
    assert topk(lib, stride=63) == EINVAL
    assert topk(lib, rows=-1) == EINVAL
    assert topk(lib, out_idx=None) == EINVAL
    assert topk(lib, out_idx_stride=4) == EINVAL
    assert topk(lib, want_values=1) == EINVAL          # no value buffer
    assert topk(lib, x=FAKE + 8) == EALIGN              # base not on 16 bytes
    assert topk(lib, cols=65, stride=65) == EALIGN      # 260-byte rows
    assert topk(lib, dtype=1, cols=60, stride=60) == EALIGN
    assert topk(lib, out_idx_stride=9) == EALIGN        # 36-byte output rows
    assert topk(lib, sorted_index=3) == EINVAL          # SEL_UNSORTED / SEL_SORT_INDEX / SEL_SORT_VALUE only
    assert topk(lib, sorted_index=-1) == EINVAL
    assert topk(lib, rows=0) == 0                       # nothing to do, no launch
    assert topk(lib, rows=0, sorted_index=2) == 0


def test_workspace_size_rejects_bad_arguments(lib):
    # invalid shapes answer 0 without touching the device
    assert lib.sel_topk_workspace_size(7, 4, 64, 8) == 0
    assert lib.sel_topk_workspace_size(0, 4, 64, 0) == 0
    assert lib.sel_topk_workspace_size(0, 4, 64, 5000) == 0
    assert lib.sel_topk_workspace_size(0, 0, 64, 8) == 0


def test_kernel_name_rejects_bad_arguments(lib):
    # invalid shapes answer NULL without touching the device
    assert lib.sel_topk_kernel_name(7, 4, 64, 8, 0) is None
    assert lib.sel_topk_kernel_name(0, 4, 64, 0, 0) is None
    assert lib.sel_topk_kernel_name(1, 4, 64, 8, 9) is None
    assert lib.sel_topk_kernel_name(1, 4, 64, 8, -1) is None


def test_gather_rejections(lib):
    EINVAL, EALIGN = 1, 2
    def g(key=FAKE, b=1, comp_len=10, d=64, kbs=640, krs=64, idx=FAKE, idx_dtype=0, rows=4, n=3, irs=3, out=FAKE):
        return lib.sel_gather_rows(key, b, comp_len, d, kbs, krs, idx, idx_dtype, rows, n, irs, out, None, None)
    assert g(d=12, krs=12, kbs=120) == EALIGN
    assert g(rows=5, b=2) == EINVAL
    assert g(idx=None) == EINVAL
    assert g(idx_dtype=2) == EINVAL
    assert g(krs=32) == EINVAL  # row stride < d
    assert g(key=FAKE + 2) == EALIGN
    assert g(rows=0) == 0 and g(n=0) == 0


def test_gather_pair_rejections(lib):
    EINVAL, EALIGN = 1, 2
    def g(key=FAKE, d=64, kbs=640, krs=64, key2=FAKE, d2=256, kbs2=2560, krs2=256, b=1, comp_len=10, idx=FAKE,
          idx_dtype=0, rows=4, n=3, irs=3, out=FAKE, out2=FAKE):
        return lib.sel_gather_rows_pair(key, d, kbs, krs, key2, d2, kbs2, krs2, b, comp_len, idx, idx_dtype, rows,
                                        n, irs, out, out2, None, None)
    assert g(d2=12, krs2=12, kbs2=120) == EALIGN   # second key rows not whole 16-byte vectors
    assert g(krs2=128) == EINVAL                   # second key row stride < d2
    assert g(key2=None) == EINVAL
    assert g(out2=None) == EINVAL
    assert g(key2=FAKE + 2) == EALIGN
    assert g(rows=5, b=2) == EINVAL
    assert g(idx_dtype=2) == EINVAL
    assert g(rows=0) == 0 and g(n=0) == 0


def test_block_rejections(lib):
    EINVAL, EALIGN, EUNSUP = 1, 2, 3
    def g(scores=FAKE, rows=4, n_blocks=32, stride=32, tb=4, bs=64, out_pos=FAKE, ops=256, key=None, b=1,
          comp_len=2048, d=128, kbs=2048 * 128, krs=128, gout=None):
        return lib.sel_block_topk_gather(scores, 0, rows, n_blocks, stride, None, tb, bs, out_pos, ops, key, b,
                                         comp_len, d, kbs, krs, gout, None, 0, None, None, None)
    assert g(bs=0) == EINVAL
    assert g(tb=0) == EINVAL
    assert g(tb=4097) == EINVAL
    assert g(ops=252) == EINVAL            # out_pos rows shorter than topk_blocks * block_size
    assert g(ops=258) == EALIGN            # 1032-byte rows
    assert g(out_pos=None) == EINVAL
    assert g(key=FAKE) == EINVAL           # key without an output
    assert g(gout=FAKE) == EINVAL          # output without a key
    assert g(key=FAKE, gout=FAKE, d=12, krs=12, kbs=12 * 2048) == EALIGN
    assert g(n_blocks=1 << 20, stride=1 << 20, bs=1 << 12) == EUNSUP   # positions past int32
    assert g(rows=0) == 0


def test_fused_rejections(lib):
    r = lib.sel_topk_gather(FAKE, 0, 4, 64, 64, None, 8, 0, 0, 0, None, 0, None, 0,
                            FAKE, 1, 64, 64, 64 * 64, 64, 9, FAKE, None, 0, None, None, None)
    assert r == 1  # n_gather > k
    r = lib.sel_topk_gather(FAKE, 0, 4, 64, 64, None, 8, 0, 0, 0, None, 0, None, 0,
                            FAKE, 3, 64, 64, 64 * 64, 64, 8, FAKE, None, 0, None, None, None)
    assert r == 1  # rows not a multiple of b
    r = lib.sel_topk_gather(FAKE, 0, 4, 64, 64, None, 8, 2, 0, 0, None, 0, None, 0,
                            FAKE, 1, 64, 64, 64 * 64, 64, 8, FAKE, None, 0, None, None, None)
    assert r == 1  # value order gathers from the index rows, so out_idx is required
    r = lib.sel_topk_gather(FAKE, 0, 4, 64, 64, None, 8, 5, 0, 0, FAKE, 8, None, 0,
                            FAKE, 1, 64, 64, 64 * 64, 64, 8, FAKE, None, 0, None, None, None)
    assert r == 1  # bad order


def test_product_has_no_cpu_path():
    """The package imports no oracle code and fails loudly without its library."""
    import gather_radix_select_gb300 as g
    from gather_radix_select_gb300 import _native
    pkg = os.path.dirname(g.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle/" not in text, f
    saved = _native._lib
    real = _native.library_path
    try:
        _native._lib = None
        _native.library_path = lambda: "/nonexistent/libsel.so"
        with pytest.raises(RuntimeError):
            _native.load()
    finally:
        _native.library_path = real
        _native._lib = saved
