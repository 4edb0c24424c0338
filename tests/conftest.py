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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running statistical test")


@pytest.fixture(scope="session")
def built_library():
    """Path of the compiled C-ABI library, building it in-tree if it is missing."""
    from speculative_decoding_token_temperature_gb300 import build as _build
    return _build.ensure_built()


@pytest.fixture
def hooks(built_library):
    """Set library test hooks for one test (hooks(name=value, ...)); restored afterwards."""
    import speculative_decoding_token_temperature_gb300 as sd
    guards = []

    def set_hooks(**kw):
        g = sd.test_hooks(**kw)
        g.__enter__()
        guards.append(g)

    yield set_hooks
    for g in reversed(guards):
        g.__exit__(None, None, None)
