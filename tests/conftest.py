import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: a CPU test that takes more than a few seconds")


def _figures():
    path = os.path.join(ROOT, "tests", "golden", "pages_figures.txt")
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            name, rest = line.split("=", 1)
            value = rest.split(";", 1)[0].strip()
            out[name.strip()] = float(value) if any(c in value for c in ".e") else int(value)
    return out


FIGURES = _figures()


@pytest.fixture(scope="session")
def figures():
    return FIGURES
