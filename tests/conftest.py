import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def read_golden(name):
    """Parse a golden fixture: 'key = values' lines and bare numeric rows; '#' starts a comment."""
    kv, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if "=" in line:
                k, v = line.split("=", 1)
                kv[k.strip()] = [float(t) for t in v.split()]
            else:
                rows.append([float(t) for t in line.split()])
    return kv, rows


@pytest.fixture
def golden():
    return read_golden
