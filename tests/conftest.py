import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden_path(name: str) -> str:
    return os.path.join(ROOT, "tests", "golden", name)


def read_golden(name: str):
    """Parse a fixture: '#' lines are comments; 'key = value' lines or raw rows."""
    kv, rows = {}, []
    with open(golden_path(name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if " = " in line:
                k, v = line.split(" = ", 1)
                kv.setdefault(k.strip(), []).append(v.strip())
            else:
                rows.append(line.split())
    return kv, rows
