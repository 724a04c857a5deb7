import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); run on the GPU host")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _device_error_word(request):
    """After every GPU test: zero_sync() must report no device-side error (a
    bounded wait that gave up, or, in a bounds-checked build, an index that
    fell outside its buffer)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    try:
        import torch
    except ImportError:
        return
    if not torch.cuda.is_available():
        return
    from zero_sharded_optimizer_flatten_gb300 import zero as Z
    if Z._lib is None:
        return
    Z.zero_sync()
