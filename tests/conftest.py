import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large full-size parity case")


@pytest.fixture(scope="session")
def orc():
    from oracle import oracle
    oracle.build()
    return oracle


def pytest_sessionfinish(session, exitstatus):
    """With RA_PARITY_REPORT set, write the errors the parity tests measured
    (max-abs and relative, per output) to that file as JSON."""
    path = os.environ.get("RA_PARITY_REPORT")
    mod = sys.modules.get("parity_util")
    if not path or mod is None or not mod.RECORDS:
        return
    with open(path, "w") as f:
        json.dump(mod.RECORDS, f, indent=1, sort_keys=True)
