import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _no_failed_device_checks(request):
    """With the debug build loaded (WKV7_LIBRARY names libwkv7_debug.so), every GPU test must leave the
    device-side index checks clean."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import linear_rnn_lm_wkv7_b300 as wkv7
    if wkv7.debug_enabled():
        assert wkv7.debug_status() == 0, "a device-side index check failed"
