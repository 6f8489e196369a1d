import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # a gpu-marked test on a machine without a GPU is a skip, never a silent CPU run
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture
def tuning():
    """set_tuning for one test: forces a kernel plan (plan="wide", parts=7, ...) and puts every
    knob back afterwards."""
    import gather_radix_select_gb300 as g
    saved = g.get_tuning()
    yield g.set_tuning
    g.set_tuning(**saved)
