import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(autouse=True)
def _parity_test_name(request):
    try:
        import hstu_testutil
    except Exception:  # CPU-only runs without the helpers' imports
        yield
        return
    hstu_testutil.CURRENT_TEST["name"] = request.node.nodeid
    yield


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("HSTU_PARITY_LOG")
    if not path:
        return
    try:
        import hstu_testutil
    except Exception:
        return
    if not hstu_testutil.MARGINS:
        return
    import json
    with open(path, "w") as f:
        json.dump(hstu_testutil.MARGINS, f, indent=0)
