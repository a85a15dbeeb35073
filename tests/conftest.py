import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def golden():
    """tests/golden/worked_examples.txt as {id: (inputs, expected, source)}."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", "worked_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ident, inp, exp, src = [p.strip() for p in line.split(";", 3)]
            parse = lambda s: [] if s == "-" else [float(t) for t in s.split()]
            out[ident] = (parse(inp), parse(exp), src)
    return out
