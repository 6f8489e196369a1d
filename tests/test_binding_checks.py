"""The Python binding's checks of caller-owned output buffers (no GPU: pure tensor checks)."""
import pytest
import torch


def test_output_index_buffer_checks():
    import gather_radix_select_gb300 as g
    cpu = torch.device("cpu")
    ok = torch.empty((3, 8), dtype=torch.int64)
    assert g._out_idx(ok, 3, 8, torch.int64, cpu) is ok
    assert g._out_idx(None, 3, 5, torch.int32, cpu).shape == (3, 5)
    with pytest.raises(ValueError):
        g._out_idx(torch.empty((3, 8), dtype=torch.int32), 3, 8, torch.int64, cpu)  # 4-byte rows for 8-byte indices
    with pytest.raises(ValueError):
        g._out_idx(torch.empty((3, 7), dtype=torch.int64), 3, 8, torch.int64, cpu)  # shorter than k
    with pytest.raises(ValueError):
        g._out_idx(torch.empty((2, 8), dtype=torch.int64), 3, 8, torch.int64, cpu)  # too few rows
    with pytest.raises(ValueError):
        g._out_idx(torch.empty((8, 3), dtype=torch.int64).t(), 3, 8, torch.int64, cpu)  # strided rows
    with pytest.raises(TypeError):
        g._out_idx(None, 3, 8, torch.int16, cpu)


def test_output_value_buffer_checks():
    import gather_radix_select_gb300 as g
    cpu = torch.device("cpu")
    ok = torch.empty((4, 16), dtype=torch.bfloat16)
    assert g._out_val(ok, 4, 10, torch.bfloat16, cpu) is ok
    with pytest.raises(ValueError):
        g._out_val(torch.empty((4, 16), dtype=torch.float32), 4, 10, torch.bfloat16, cpu)
    with pytest.raises(ValueError):
        g._out_val(torch.empty((4, 9), dtype=torch.bfloat16), 4, 10, torch.bfloat16, cpu)
