import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libfp4gemv.so")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _device_error_word_clear(request):
    """After every GPU test: the library's device error word (a bounded wait
    that ran out, a bad expert id) must be clear.  Tests that provoke an error
    read and clear it themselves."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    mod = sys.modules.get("moe_nvfp4_gemv_gb300.fp4gemv")
    if mod is None or getattr(mod, "_lib", None) is None:
        return
    code = mod.get_device_error()
    assert code == 0, f"device error word {code} after {request.node.nodeid}"
