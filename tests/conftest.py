import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Parse a whitespace text fixture: '#' comments, then 'tag values...'."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            rows.append((tag, vals))
    return rows


def golden_eps(cfg):
    """eps of synthetic workload cfg (written by tests/golden/make_eps.py)."""
    import json
    with open(os.path.join(GOLDEN, "eps_configs.json")) as f:
        return json.load(f)[str(cfg)]["eps"]
