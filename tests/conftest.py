import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture
def tune():
    """Planner overrides for one test: ``tune(gemm_pair=0)`` sets knobs
    through rarn_set_tuning; every knob is reset when the test ends."""
    import residual_add_rmsnorm_gb300 as rarn

    def set_knobs(**knobs):
        for k, v in knobs.items():
            rarn.set_tuning(k, v)

    try:
        yield set_knobs
    finally:
        rarn.reset_tuning()


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover - torch missing
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
