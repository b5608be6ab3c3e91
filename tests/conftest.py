import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the kernels)")
    config.addinivalue_line("markers", "slow: larger CPU cases")


def read_golden(name):
    """Non-comment lines of a golden fixture."""
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.rstrip("\n") for ln in f if ln.strip() and not ln.startswith("#")]


@pytest.fixture(scope="session")
def golden():
    return read_golden


def _ensure_library():
    """Build libvr.so for this machine before any test imports the binding."""
    from double_binary_tree_gb300 import build as _b
    _b.build(debug=True)


_ensure_library()
