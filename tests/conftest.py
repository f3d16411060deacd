import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300); parity and device tests")


def golden(name):
    """Parsed lines of a fixture under tests/golden: list of whitespace-split fields."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


@pytest.fixture(scope="session")
def ora():
    import oracle
    oracle.build()
    return oracle
