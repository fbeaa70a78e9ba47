import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 GPU and the built CUDA library")


def read_golden(name):
    """Parse a `key value` fixture (lines starting with # are the citation)."""
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(None, 1)
            vals[k] = float(v) if "." in v or "e" in v else int(v)
    return vals


@pytest.fixture(scope="session")
def golden():
    return read_golden


@pytest.fixture(scope="session")
def moe_lib():
    """The CUDA library's binding; builds libmoe.so in-tree first if it is missing."""
    from expert_routing_router_b300 import build as _b
    lib_path = os.path.join(ROOT, "expert_routing_router_b300", "libmoe.so")
    if not os.path.exists(lib_path):
        _b.build()
    from expert_routing_router_b300 import moe
    return moe
