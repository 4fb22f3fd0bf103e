import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests need a device; without one they are reported as skipped, never
    # silently routed elsewhere.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def dev():
    """cuda:0 with the library built; GPU tests only."""
    import torch
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from _util import ensure_built
    ensure_built()
    import tree_verified_block_gb300 as g
    g.lib()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    g.reset_device_status()
    return d


@pytest.fixture()
def clean_status(dev):
    """Fails the test if a kernel raised the device status word."""
    import tree_verified_block_gb300 as g
    g.reset_device_status()
    yield
    code, text = g.device_status()
    g.reset_device_status()
    assert code == 0, f"device status word set: {text}"
