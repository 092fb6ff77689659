import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


@pytest.fixture(scope="session")
def sga_lib():
    """The built C-ABI library (built in-tree if missing or stale)."""
    from greedy_spec_decode_gb300 import build as sga_build
    sga_build.build()
    import greedy_spec_decode_gb300 as sga
    return sga
