import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line(
        "markers", "slow: takes more than a few seconds")


def _gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def _built_library(request):
    """Build the CUDA library (no-op when it is up to date) before any test
    that loads it; a fresh checkout or a new machine then needs no separate step."""
    if any("gpu" in item.keywords or "test_abi" in item.nodeid
           for item in request.session.items):
        from exact_attention_forward_04_gb300 import _build
        _build.build()
