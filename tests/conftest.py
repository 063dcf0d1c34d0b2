import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree for sm_103a if it is missing or stale."""
    from paged_kv_cache_295_gb300 import _build
    _build.build_library()
    import paged_kv_cache_295_gb300 as pkv
    return pkv
