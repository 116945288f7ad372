import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def load_golden(name):
    """Read a tests/golden/<name>.txt fixture: {key: (value, tolerance)}.

    Each non-comment line is "key value printed_decimals"; the tolerance is
    half a unit in the last printed place.
    """
    path = os.path.join(ROOT, "tests", "golden", name + ".txt")
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val, dec = line.split()
            out[key] = (float(val), 0.5 * 10.0 ** (-int(dec)))
    return out


@pytest.fixture
def golden():
    return load_golden
