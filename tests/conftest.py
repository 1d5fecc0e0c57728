import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


@pytest.fixture(scope="session")
def kvc():
    """The product binding with libkvc.so built in place (nvcc cross-compiles without a GPU)."""
    from paged_kv_cache_157_gb300 import build_lib
    build_lib.build()
    import paged_kv_cache_157_gb300 as k
    k.raw()
    return k
