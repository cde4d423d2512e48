import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))
TESTS = Path(__file__).resolve().parent
if str(TESTS) not in sys.path:
    sys.path.insert(0, str(TESTS))


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


@pytest.fixture(autouse=True)
def _gpu_ready(request):
    """GPU tests need a CUDA device and the built library; fail loudly
    (never skip to a fallback) when either is missing."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import torch
    from paged_kv_cache_48_gb300 import _native
    assert torch.cuda.is_available(), "gpu test without a CUDA device"
    _native.lib()
    yield
    torch.cuda.synchronize()
