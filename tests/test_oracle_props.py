"""Property-based pins of the oracle (no GPU): random tiny rows with ties, signed zeros and
infinities, against the O(n^2) rank definition of top-k and a stable descending sort."""
import numpy as np
import pytest
import torch

import oracle

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

VALUES = st.sampled_from([0.0, -0.0, 1.0, -1.0, 0.5, 2.0, -2.5, np.inf, -np.inf, 3.0, 3.0, 1.0])


@settings(max_examples=300, deadline=None)
@given(vals=st.lists(VALUES, min_size=1, max_size=40), k=st.integers(1, 45), cut=st.integers(-3, 45),
       dtype=st.sampled_from(["f32", "bf16"]))
def test_index_order_is_the_rank_definition(vals, k, cut, dtype):
    v = np.asarray(vals, dtype=np.float32)
    bits = v.view(np.uint32) if dtype == "f32" else (v.view(np.uint32) >> 16).astype(np.uint16)
    n = len(v)
    idx, out_bits, nan = oracle.topk(bits[None, :].copy(), dtype, k, row_end=np.array([cut], np.int32),
                                     sorted_index=True)
    nv = min(max(cut, 0), n)
    want = oracle.brute_topk_row(oracle.bits_to_values(bits, dtype), nv, k)
    m = min(nv, k)
    assert idx[0][:m].tolist() == want
    assert (idx[0][m:] == -1).all()
    assert (out_bits[0][:m] == bits[want]).all()
    assert nan[0] == 0


@settings(max_examples=300, deadline=None)
@given(vals=st.lists(VALUES, min_size=1, max_size=40), k=st.integers(1, 45), cut=st.integers(-3, 45))
def test_value_order_is_a_stable_descending_sort(vals, k, cut):
    v = np.asarray(vals, dtype=np.float32)
    n = len(v)
    idx, _, _ = oracle.topk(v.view(np.uint32)[None, :].copy(), "f32", k, row_end=np.array([cut], np.int32),
                            sorted_value=True)
    nv = min(max(cut, 0), n)
    order = torch.sort(torch.from_numpy(v[:nv]), descending=True, stable=True).indices[:k].tolist()
    assert idx[0].tolist() == order + [-1] * (k - len(order))
