import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Parse a golden fixture: '#' comments; 'key: values' lines (repeated keys append);
    bare numeric lines are collected under the key 'rows'."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                out.setdefault(k.strip(), []).append(v.split())
            else:
                out.setdefault("rows", []).append(line.split())
    return out


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (built in-tree on first use)."""
    import __graft_entry__ as ge
    ge.build_library()
    from decode_gemv_epilogue_gb300 import gemvfuse
    return gemvfuse
