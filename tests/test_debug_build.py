"""The bounds-checked debug build (libsel_debug.so, SEL_LIBRARY=debug).

compute-sanitizer is not available where these kernels run, so the library
has a second build whose kernels check their own accesses: staged-list and
region offsets, workspace slots, output positions and gathered key rows.  An
access that would leave its buffer is skipped and SEL_EBOUNDS goes to
err_flag; nothing traps.  The edge-shape suites run against that build here,
in a child process (the library is chosen when it is first loaded); their
own assertions that err_flag stays 0 (or holds the expected status) then
also prove that no check fired.
"""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _debug_lib():
    from gather_radix_select_gb300 import _native, build
    if not os.path.exists(build.DEBUG_SO):
        build.build(debug=True)
    lib = ctypes.CDLL(build.DEBUG_SO)
    return lib, _native


def test_debug_library_loads_says_so_and_exports_the_boundary():
    lib, _native = _debug_lib()
    lib.sel_debug_build.restype = ctypes.c_int
    assert lib.sel_debug_build() == 1
    assert _native.load().sel_debug_build() in (0, 1)
    from tests.test_abi import declared_symbols
    for name in declared_symbols():
        assert hasattr(lib, name), name
    lib.sel_strerror.restype = ctypes.c_char_p
    assert b"debug" in lib.sel_strerror(_native.SEL_EBOUNDS)


def test_the_selected_library_follows_sel_library():
    code = ("import gather_radix_select_gb300._native as n, os; "
            "print(os.path.basename(n.library_path()), n.load().sel_debug_build())")
    env = dict(os.environ, SEL_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["libsel_debug.so", "1"]


@pytest.mark.gpu
def test_edge_shape_suites_under_the_bounds_checked_build():
    suites = ["tests/test_kernels.py", "tests/test_topk.py", "tests/test_gather.py", "tests/test_block.py",
              "tests/test_order.py", "tests/test_failure_detection.py"]
    env = dict(os.environ, SEL_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *suites],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
