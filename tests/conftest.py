import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _canary_guards():
    """After every test: the guard bytes around every canary-guarded device
    buffer (tests/guard.py) are intact."""
    yield
    import guard
    guard.check_guards()
