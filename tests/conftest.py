import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size case, minutes of CPU or GPU time")


def read_golden(name):
    """Parse a tests/golden/*.txt fixture: 'key = v1 v2 ...' lines (ints, or floats where written
    with a point or exponent), '#' comments."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition("=")
            out[key.strip()] = [float(v) if any(c in v for c in ".eE") else int(v) for v in val.split()]
    return out
