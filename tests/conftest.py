import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large inputs")


@pytest.fixture(autouse=True)
def _parity_test_name(request):
    import parity

    parity._CURRENT["test"] = request.node.nodeid
    yield


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("TACO_PARITY_REPORT")
    if not path:
        return
    import json

    import parity

    with open(path, "w") as f:
        json.dump(parity.REPORT, f, indent=1, sort_keys=True)
