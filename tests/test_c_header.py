"""The boundary from plain C: include/sel.h compiles as C99 with warnings as errors, a C program
links against libsel.so, and the host-side argument checks answer without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "sel.h"
#include "sel_tuning.h"

int main(void)
{
    int in_align = 0, out_align = 0;
    if (sel_stride_requirement(&in_align, &out_align) != SEL_OK || in_align != 16 || out_align != 16) return 1;
    /* k out of range, value order without indices, an unknown order: refused before any CUDA call */
    char x[64] __attribute__((aligned(16)));
    int idx[16] __attribute__((aligned(16)));
    if (sel_topk(x, SEL_F32, 1, 16, 16, NULL, 0, SEL_UNSORTED, SEL_I32, 0, idx, 16, NULL, 0, NULL, 0, NULL, NULL,
                 NULL) != SEL_EINVAL) return 2;
    if (sel_topk(x, SEL_F32, 1, 16, 16, NULL, 4, 3, SEL_I32, 0, idx, 16, NULL, 0, NULL, 0, NULL, NULL,
                 NULL) != SEL_EINVAL) return 3;
    if (sel_topk(x, SEL_BF16, 0, 16, 16, NULL, 4, SEL_SORT_VALUE, SEL_I64, 0, idx, 16, NULL, 0, NULL, 0, NULL,
                 NULL, NULL) != SEL_OK) return 4;  /* no rows: nothing to do */
    if (sel_gather_rows(x, 1, 4, 12, 48, 12, idx, SEL_I32, 1, 1, 1, x, NULL, NULL) != SEL_EALIGN) return 5;
    if (sel_block_topk_gather(x, SEL_F32, 1, 16, 16, NULL, 4, 0, idx, 16, NULL, 1, 0, 0, 0, 0, NULL, NULL, 0,
                              NULL, NULL, NULL) != SEL_EINVAL) return 6;  /* block_size 0 */
    if (sel_max_cols(SEL_BF16) <= 0 || sel_topk_workspace_size(7, 1, 16, 4) != 0) return 7;
    /* the tuning knobs: set, read back, restore */
    {
        const int plan = sel_get_tuning(SEL_TUNE_PLAN);
        if (sel_set_tuning(SEL_TUNE_PLAN, SEL_PLAN_FLAT) != SEL_OK || sel_get_tuning(SEL_TUNE_PLAN) != SEL_PLAN_FLAT)
            return 8;
        if (sel_set_tuning(SEL_TUNE_PLAN, plan) != SEL_OK || sel_set_tuning(99, 0) != SEL_EINVAL) return 9;
    }
    printf("%s\n", sel_strerror(SEL_EALIGN));
    return 0;
}
"""


def test_header_is_c99_and_the_library_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from gather_radix_select_gb300 import _native
    so = _native.library_path()
    if not os.path.exists(so):
        from gather_radix_select_gb300 import build
        build.build()
    src = tmp_path / "use_sel.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_sel"
    libdir = os.path.dirname(so)
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(src), "-o", str(exe), so, "-Wl,-rpath," + libdir])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.strip()
