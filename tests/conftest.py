import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def mmlib():
    """The built C-ABI library (built in-tree if missing or stale)."""
    from mixture_experts_layer_mm_gb300 import buildlib
    import mixture_experts_layer_mm_gb300 as pkg
    buildlib.build()
    pkg.lib()
    return pkg
