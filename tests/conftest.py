import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    # GPU tests run only where a GPU exists; a GPU machine without the built
    # library fails loudly inside the tests instead of skipping.
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


@pytest.fixture(autouse=True)
def _device_buffer_guards(request):
    """After every GPU test: no canary guard around a device buffer of the
    test's layers (pages, tables, descriptors, workspaces) has changed."""
    yield
    if "gpu" not in request.keywords:
        return
    import _layers
    bad = []
    for m in _layers.LIVE:
        bad.extend(m.corrupted_guards())
    _layers.LIVE.clear()
    assert not bad, f"device buffer guards overwritten: {bad[:8]}"
