import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Parse a ``key = value`` fixture under tests/golden (``#`` lines are comments)."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = [s.strip() for s in line.split("=", 1)]
            parts = v.split()
            vals = []
            for p in parts:
                try:
                    vals.append(int(p))
                except ValueError:
                    vals.append(float(p))
            out[k] = vals[0] if len(vals) == 1 else vals
    return out
