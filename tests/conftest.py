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
