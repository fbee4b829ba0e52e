import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    from oracle import oracle as o
    o.build()
    return o


@pytest.fixture(scope="session")
def gemm_mod():
    """The ctypes binding, building the library first if needed."""
    from dense_gemm_row_gb300 import build as b
    b.build(quiet=True)
    from dense_gemm_row_gb300 import binding as g
    return g
