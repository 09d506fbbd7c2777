import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")
    config.addinivalue_line("markers", "timing: asserts on measured GPU times (collected after every other test)")


def pytest_collection_modifyitems(config, items):
    # Tests that assert on measured times depend on the box they run on; run them
    # after the parity tests, so that under -x a slow box stops no parity check.
    timed = [it for it in items if it.get_closest_marker("timing")]
    if timed:
        items[:] = [it for it in items if not it.get_closest_marker("timing")] + timed


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture
def load_golden():
    return golden
