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
    """Non-comment lines of a golden fixture, split on ':' into (key, values)."""
    out = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                out.append((k.strip(), v.split()))
            else:
                out.append((line, []))
    return out


@pytest.fixture(scope="session", autouse=True)
def _native_library(request):
    """Build libdsa_rr.so once per session when GPU tests are collected (a no-op when fresh)."""
    if any(item.get_closest_marker("gpu") for item in request.session.items):
        from deepseek_v3_sparse_round_gb300 import build as b
        b.build()
    yield
