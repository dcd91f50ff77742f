import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden(name):
    """Parse a tests/golden fixture: '# ...' comments, 'key: values' lines and
    bare rows of numbers.  Returns (dict of key -> list of str, list of rows)."""
    kv, rows = {}, []
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                key, val = line.split(":", 1)
                kv[key.strip()] = val.split()
            else:
                rows.append(line.split())
    return kv, rows
