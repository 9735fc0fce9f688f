import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built libgsr.so")
    config.addinivalue_line("markers", "slow: large CPU oracle runs")


def golden(name):
    return os.path.join(ROOT, "tests", "golden", name)


def read_page_constants():
    rows = []
    with open(golden("page_constants.txt")) as f:
        for line in f:
            line = line.split("--")[0].strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((parts[0], float(parts[1]), float(parts[2]) if len(parts) > 2 else None))
    return rows
