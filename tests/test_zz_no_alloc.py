"""sel_topk_noalloc: top-k for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace -- a framework may already
own every byte of the device pool, or the caller may be plain C code with no
device allocator.  sel_topk_noalloc takes its scratch from an array built
into the library instead.  These tests call it through the C ABI and check
that it returns exactly what sel_topk with a caller workspace returns, on two
calls in a row (the array keeps the previous call's contents, so the second
call checks that nothing stale leaks through).  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic as syn

pytestmark = pytest.mark.gpu


def lib():
    from gather_radix_select_gb300 import _native
    return _native.load()


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def padded(rows, k, dtype):
    per = 16 // torch.empty((), dtype=dtype).element_size()
    return torch.full((rows, (k + per - 1) // per * per), -3, dtype=dtype, device="cuda")


def run_both(x, dtype_code, rows, cols, k, idx_dtype, want_values, row_end=None, sorted_index=1):
    """sel_topk with a fresh workspace, then sel_topk_noalloc twice, with a no-alloc call on other
    data (the rows negated) in between, so that the second compared call finds the array holding
    another input's candidates.  Returns the scratch size and the three compared results."""
    from gather_radix_select_gb300 import _native
    L = lib()
    itype = torch.int64 if idx_dtype == 1 else torch.int32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    need = L.sel_topk_workspace_size(dtype_code, rows, cols, k)
    assert need <= _native.SEL_NOALLOC_SCRATCH_BYTES
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    other = -x
    results = []
    for mode in ("workspace", "noalloc", "noalloc-other", "noalloc"):
        src = other if mode == "noalloc-other" else x
        idx = padded(rows, k, itype)
        val = padded(rows, k, x.dtype) if want_values else None
        nan = torch.zeros(1, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        common = (ptr(src), dtype_code, rows, cols, src.stride(0), ptr(row_end), k, sorted_index, idx_dtype,
                  int(want_values), ptr(idx), idx.stride(0), ptr(val), 0 if val is None else val.stride(0))
        if mode == "workspace":
            st = L.sel_topk(*common, ptr(ws), ws.numel(), ptr(nan), ptr(err), stream)
        else:
            st = L.sel_topk_noalloc(*common, ptr(nan), ptr(err), stream)
        assert st == 0, L.sel_strerror(st)
        torch.cuda.synchronize()
        if mode != "noalloc-other":
            results.append((idx[:, :k].cpu(), None if val is None else val[:, :k].cpu(), int(nan.item()),
                            int(err.item())))
    return need, results


def same(a, b):
    ia, va, na, ea = a
    ib, vb, nb, eb = b
    assert torch.equal(ia, ib)
    if va is not None:
        assert torch.equal(va.view(torch.int16) if va.dtype == torch.bfloat16 else va.view(torch.int32),
                           vb.view(torch.int16) if vb.dtype == torch.bfloat16 else vb.view(torch.int32))
    assert na == nb and ea == eb == 0


def test_noalloc_matches_workspace_entry_point_on_split_rows(tuning):
    # four 204800-wide bf16 rows split over many CTAs (forced), so the scratch is really used
    tuning(plan="split")
    w = syn.workload("indexer_bf16_4x204800_k1024")
    x = torch.from_numpy(w["x"].view(np.int16)).view(torch.bfloat16).cuda()
    need, res = run_both(x, 1, w["rows"], w["cols"], w["k"], 0, True)
    assert need > 0
    same(res[0], res[1])
    same(res[0], res[2])


def test_noalloc_on_the_default_plan_of_few_wide_rows():
    # no forced plan: four 204800-wide bf16 rows are split over many CTAs whose candidate lists
    # meet in the scratch
    import oracle
    import gather_radix_select_gb300 as g
    w = syn.workload("indexer_bf16_4x204800_k1024")
    assert g.kernel_name(torch.bfloat16, w["rows"], w["cols"], w["k"]) in ("wide_kernel", "flat_kernel")
    x = torch.from_numpy(w["x"].view(np.int16)).view(torch.bfloat16).cuda()
    need, res = run_both(x, 1, w["rows"], w["cols"], w["k"], 0, True)
    assert need > 0
    same(res[0], res[1])
    same(res[0], res[2])
    o_idx, o_bits, _ = oracle.topk(w["x"], "bf16", w["k"], sorted_index=True)
    assert (res[1][0].numpy() == o_idx).all()
    assert (res[1][1].view(torch.int16).numpy().view(np.uint16) == o_bits).all()


@pytest.mark.parametrize("plan", ["split", "flat"])
def test_noalloc_matches_on_fp32_split_rows_with_row_end_and_nan(plan, tuning):
    tuning(plan=plan)
    rng = np.random.default_rng(31)
    rows, cols, k = 6, 131072, 4096
    v = (rng.standard_normal((rows, cols)) * 2).astype(np.float32)
    v[2, 777] = np.nan
    x = torch.from_numpy(v).cuda()
    end = torch.tensor([cols, 100000, cols, 5000, 3000, 0], dtype=torch.int32, device="cuda")
    need, res = run_both(x, 0, rows, cols, k, 1, True, row_end=end)
    assert need > 0
    same(res[0], res[1])
    same(res[0], res[2])
    assert res[0][2] == 1


def test_noalloc_value_order(tuning):
    # value-ordered output through the no-workspace entry point, on split rows
    tuning(plan="split")
    import oracle
    w = syn.workload("indexer_bf16_4x204800_k1024")
    x = torch.from_numpy(w["x"].view(np.int16)).view(torch.bfloat16).cuda()
    need, res = run_both(x, 1, w["rows"], w["cols"], w["k"], 1, True, sorted_index=2)
    assert need > 0
    same(res[0], res[1])
    same(res[0], res[2])
    o_idx, o_bits, _ = oracle.topk(w["x"], "bf16", w["k"], sorted_value=True)
    assert (res[1][0].numpy() == o_idx).all()
    assert (res[1][1].view(torch.int16).numpy().view(np.uint16) == o_bits).all()


def test_noalloc_without_scratch_and_oversize_rejection(tuning):
    # a shape that needs no scratch runs too
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.standard_normal((300, 2048)).astype(np.float32)).cuda()
    need, res = run_both(x, 0, 300, 2048, 64, 0, False, sorted_index=0)
    assert need == 0
    same(res[0], res[1])
    same(res[0], res[2])
    # a shape whose scratch exceeds the built-in array is refused before any launch
    tuning(plan="split")
    L = lib()
    from gather_radix_select_gb300 import _native
    rows, cols = 300, 2_000_000
    assert L.sel_topk_workspace_size(0, rows, cols, 4096) > _native.SEL_NOALLOC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    out = torch.empty((rows, 4096), dtype=torch.int32, device="cuda")
    st = L.sel_topk_noalloc(ptr(dummy), 0, rows, cols, cols, None, 4096, 0, 0, 0, ptr(out), 4096, None, 0,
                            None, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _native.SEL_ESCRATCH
    assert b"scratch" in L.sel_strerror(st)
