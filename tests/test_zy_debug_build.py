"""The edge-shape, decay and decode parity tests again on libwkv7_debug.so, the build with device-side
index checks: every kernel checks the indices it derives (shared-memory operand rows and columns, global
rows, block indices) and records a failed check instead of making the access.  The tests run in a child
process with WKV7_LIBRARY naming that build; conftest.py asserts wkv7_debug_status() == 0 after each.
(A stand-in for a device memory checker.)"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEBUG_LIB = os.path.join(ROOT, "linear_rnn_lm_wkv7_b300", "libwkv7_debug.so")


def test_debug_library_exports_the_check_entry_points():
    import ctypes
    import linear_rnn_lm_wkv7_b300 as wkv7
    assert not wkv7.debug_enabled()  # the release build is the default
    assert wkv7.lib.wkv7_debug_status(None) == 1
    if os.path.exists(DEBUG_LIB):
        dbg = ctypes.CDLL(DEBUG_LIB)
        assert dbg.wkv7_debug_enabled() == 1


@pytest.mark.gpu
def test_edge_and_decay_parity_under_device_checks():
    assert os.path.exists(DEBUG_LIB), "build libwkv7_debug.so first (python linear_rnn_lm_wkv7_b300/build.py --debug)"
    env = dict(os.environ, WKV7_LIBRARY=DEBUG_LIB)
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_parity_gpu.py"), "-q", "-x", "-m", "gpu",
           "-p", "no:cacheprovider", "-k", "edge or decay or zero_tokens or many_heads or decode_small or workspace"]
    res = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=1800)
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-2000:]
    assert " passed" in res.stdout
