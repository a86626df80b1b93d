import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libqmoe.so")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def guard_bands(request):
    """In every GPU test, each tensor the binding allocates for a kernel to write
    (outputs, padded sorted rows, scale factors, fp32 accumulation buffers) sits
    between two sentinel-filled margins; after the test every margin must be
    intact, so a store past either end of any of them fails the test."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    from tests import guard
    with guard.guarded_allocations() as check:
        yield
        check()
