import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, where no GPU is present; the CUDA
    # library itself still has to load (tests/test_abi.py checks that on CPU).
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def device_status_clear(request):
    """After every GPU test, no kernel's bounded wait may have expired (a
    kernel that gives up returns early with its outputs unfinished). The
    bounded-wait self test reads and clears the word itself."""
    yield
    if "gpu" not in request.node.keywords:
        return
    import torch

    if not torch.cuda.is_available():
        return
    import long_context_causal_blockwise_gb300 as lcb

    bits, where = lcb.take_device_status()
    assert bits == 0, f"a bounded wait expired during this test: status {bits:#x}, where {where:#x}"
