import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Parity figures gathered by the GPU tests (rows compared, selection outcome, max-abs and relative
# Frobenius error per output, oracle seconds).  Written as JSON at the end of the session when
# SDA_PARITY_REPORT names a file.
_PARITY = {}


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU check")


@pytest.fixture(scope="session")
def parity_report():
    return _PARITY


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("SDA_PARITY_REPORT")
    if path and _PARITY:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            json.dump(_PARITY, f, indent=1, sort_keys=True)
