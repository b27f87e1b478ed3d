import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_sessionfinish(session, exitstatus):
    """EP_PARITY_LOG=<file>: write every combined-output comparison (both metrics)."""
    path = os.environ.get("EP_PARITY_LOG")
    if not path:
        return
    try:
        from parity_util import PARITY_LOG
    except ImportError:
        return
    import json
    with open(path, "w") as f:
        json.dump(PARITY_LOG, f, indent=1)
