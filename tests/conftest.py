import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libcar.so")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


def read_golden(name):
    """Parse a key: value fixture; '#' lines are citations/comments.  Returns a list of case dicts."""
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            key, val = key.strip(), val.strip()
            if key == "case" and cur:
                cases.append(cur)
                cur = {}
            cur[key] = val
    if cur:
        cases.append(cur)
    return cases
