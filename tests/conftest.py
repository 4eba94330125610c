import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


def pytest_sessionstart(session):
    """Build the CUDA library (sm_103a, cross-compiled: no GPU needed) if it is missing, so that
    the suite runs on a fresh checkout.  A present library is used as it is."""
    lib = os.path.join(ROOT, "mxfp4_routed_expert_06_b300", "libk3moe.so")
    if not os.path.exists(lib):
        import importlib.util

        spec = importlib.util.spec_from_file_location(
            "k3moe_build", os.path.join(ROOT, "mxfp4_routed_expert_06_b300", "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Parse a golden fixture: '#' comments, then 'key v1 v2 ...' lines (repeated keys kept in order)."""
    out = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out.append((key, vals))
    return out


@pytest.fixture
def golden():
    return read_golden
