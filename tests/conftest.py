import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    # A child run of the suites on the checked build (tests/test_checked_build_gpu.py) names
    # that library here; it is loaded before any test loads the normal one.
    checked = os.environ.get("AQ_TEST_CHECKED_LIB")
    if checked:
        from rank_weight_reconstruction_gb300 import binding
        binding.load(checked)


def pytest_collection_modifyitems(config, items):
    # GPU tests must never run silently on a machine without a GPU: they are skipped
    # only when no CUDA device exists at all (the CPU suite deselects them anyway).
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
