"""Shared test setup: the ``gpu`` marker and in-tree builds of the libraries.

CPU tests (``-m "not gpu"``) need the oracle and the input generator built for
this machine; the C-ABI library is built too so its exports can be checked.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


def pytest_sessionstart(session):
    import oracle
    import synth
    if not os.path.exists(oracle.LIB_PATH):
        oracle.build()
    if not os.path.exists(synth.LIB_PATH):
        synth.build()
    try:
        import fsdp_sharded_mixed_gb300 as zs
    except ImportError:
        return
    if not (os.path.exists(zs.LIB_PATH) and os.path.exists(zs.CHECKED_LIB_PATH)):
        zs.build()


@pytest.fixture(autouse=True)
def _bounds_word_clear(request):
    """Under the bounds-checked library (ZS_BOUNDS_CHECK=1), every GPU test
    ends with the device error word clear: no kernel access fell outside its
    launch's window (tests that set the word on purpose read and clear it)."""
    yield
    if os.environ.get("ZS_BOUNDS_CHECK") == "1" and request.node.get_closest_marker("gpu"):
        import fsdp_sharded_mixed_gb300 as zs
        zs.zs_check_device_error()


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()
