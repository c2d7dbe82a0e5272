import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def parse_value(tok: str) -> float:
    """Golden-file value token: decimal, '-0', '2^k' or 'a*2^k'."""
    neg = tok.startswith("-")
    t = tok[1:] if neg else tok
    if "*" in t:
        a, b = t.split("*")
        v = float(a) * parse_value(b)
    elif t.startswith("2^"):
        v = 2.0 ** int(t[2:])
    else:
        v = float(t)
    return -v if neg else v


def read_records(path):
    recs = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            recs.append([p.strip() for p in line.split("|")])
    return recs


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
