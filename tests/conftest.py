import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libringattn")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def ralib():
    """The built libringattn (compiled in-tree on first use): the product
    build, or the bounds-checked / traced flavour when RA_DEBUG / RA_TRACE is
    1 (the binding loads that one)."""
    from ring_chunked_attention_gb300 import build as b

    b.build()
    import ring_chunked_attention_gb300 as ra

    if ra._DEBUG or ra._TRACE:
        b.build(debug=ra._DEBUG, trace=ra._TRACE)
    ra._load()
    return ra


@pytest.fixture(scope="session")
def cuda_ok():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True
