import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--bounds-checked", action="store_true",
                     help="run every test through the bounds-checked library (build(debug=True)): a computed "
                          "index outside its buffer then sets ORPO_STATUS_BOUNDS, which the tests' status "
                          "checks report")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU-side oracle work")
    if config.getoption("--bounds-checked"):
        import orpo_preference_loss_gb300 as orpo
        from orpo_preference_loss_gb300 import build
        build.build(debug=True)
        orpo.use_bounds_checked_library()


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
