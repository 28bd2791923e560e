import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def golden_path(name):
    return os.path.join(GOLDEN, name)


def read_kv_golden(name):
    """Parse a 'key = value  # comment' golden file into a dict of strings."""
    out = {}
    with open(golden_path(name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = [s.strip() for s in line.split("=", 1)]
            out[k] = v
    return out


@pytest.fixture
def golden():
    return read_kv_golden
