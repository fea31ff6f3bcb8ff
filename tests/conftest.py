import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large full-size parity case")


def has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


def pytest_collection_modifyitems(config, items):
    if has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _device_error_word_stays_clear(request):
    """Every GPU test leaves the library's device error word clear: a bounded
    wait that ran out inside a kernel (or invalid device data) fails the test
    that caused it, even when that test's outputs happened to be right."""
    yield
    if request.node.get_closest_marker("gpu") is None or not has_gpu():
        return
    import exact_attention_tiled_gb300 as fa
    st, site = fa.fa_device_error(clear=True)
    assert st == 0, f"device error word set during {request.node.name}: status {st}, site {site:#x}"
