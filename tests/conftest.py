import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")
    config.addinivalue_line("markers", "cpu: runs without a GPU")


def read_golden(name):
    """Rows of a golden fixture: comment lines ('#') skipped, fields split."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def golden_orders(name):
    """{chunk: [ranks in accumulation order]} from an order fixture."""
    out = {}
    for row in read_golden(name):
        assert row[0] == "chunk" and row[2] == "order"
        out[int(row[1])] = [int(v) for v in row[3:]]
    return out
