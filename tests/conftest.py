import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity cases (minutes of CPU oracle time)")


def read_golden(name):
    """Rows of a golden fixture, comments and blank lines skipped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def parse_float(tok):
    if tok in ("inf", "+inf"):
        return float("inf")
    if tok == "-inf":
        return float("-inf")
    if "0x" in tok:
        return float.fromhex(tok)
    return float(tok)
