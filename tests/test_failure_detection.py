"""Failure detection on the GPU without a fault: a bounded device wait runs out.

The tutorial's kernel calls trap() when it meets a NaN ("Speed up PyTorch
TopK with DeepSelect", "NaN handling").  This library never traps: NaNs set a
flag, and every wait of a CTA on an mbarrier (bulk copies landing in shared
memory) gives up after a bound and writes SEL_ETIMEOUT to the caller's
err_flag.  Here a self-test CTA waits, with a budget of a few microseconds, on
a barrier armed for bytes that no copy delivers; the call must come back with
err_flag == SEL_ETIMEOUT, and the next ordinary call on the same stream must
be correct.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu

SEL_ETIMEOUT = 5


def test_bounded_wait_runs_out_and_the_stream_stays_usable():
    import gather_radix_select_gb300 as g
    from gather_radix_select_gb300 import _native
    lib = _native.load()
    stream = torch.cuda.current_stream()
    for cycles in (20_000, 200_000):  # about 10 us and 100 us at 2 GHz
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = lib.sel_selftest_wait_timeout(ctypes.c_void_p(err.data_ptr()), cycles, ctypes.c_void_p(stream.cuda_stream))
        assert st == 0
        torch.cuda.synchronize()
        assert int(err.item()) == SEL_ETIMEOUT
    # the same stream then runs an ordinary selection whose rows arrive by bulk copies (the
    # staged row kernel waits on the same kind of barrier), correctly and without a timeout
    w = syn.workload("sampling_f32_4x8192_k64")
    x = torch.from_numpy(w["x"].view(np.int32)).view(torch.float32).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx = g.topk(x, w["k"], sorted_index=True, err_flag=err)
    torch.cuda.synchronize()
    assert g.kernel_name(torch.float32, w["rows"], w["cols"], w["k"]) == "row_kernel"
    assert int(err.item()) == 0
    o_idx, o_bits, _ = oracle.topk(w["x"], "f32", w["k"], sorted_index=True)
    assert (idx.cpu().numpy() == o_idx).all()
    assert (vals.contiguous().cpu().view(torch.int32).numpy().view(np.uint32) == o_bits).all()
