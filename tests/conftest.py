import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large parity cases")


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("NSM_PARITY_LOG")
    if not path:
        return
    import json

    import parity_log
    with open(path, "w") as f:
        json.dump(parity_log.RECORDS, f, indent=1)


@pytest.fixture(autouse=True)
def _device_status_clear_after_gpu_test(request):
    """After every GPU test, the device status word must read clear: no bounded wait
    expired and (in the checked build) no bounds test failed during the test, whether or
    not the test read the status itself.  Tests that make the status fire on purpose
    read it back, which clears it."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import newton_schulz_orthogonalized_gb300 as nsm
    if nsm._lib is None:  # the test never loaded the library
        return
    status = nsm.device_status_detail()
    assert status == (nsm.NSM_OK, 0, 0, 0), f"device status after the test: {status}"
