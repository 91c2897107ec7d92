"""The checked (RA_DEBUG) and traced (RA_TRACE) flavours of the library build
here without a GPU, export the same C ABI and say which flavour they are; the
product build says it is neither and refuses ra_trace_read.  (Their kernels
run in tests/test_debug_gpu.py and tests/test_trace_gpu.py.)"""
import ctypes

import pytest

from tests.test_capi import _declared_functions


@pytest.mark.parametrize("flavour,flag", [("debug", 1), ("trace", 2)])
def test_flavour_builds_and_reports_itself(ralib, flavour, flag):
    from ring_chunked_attention_gb300 import build as rab

    path = rab.build(**{flavour: True})
    lib = ctypes.CDLL(path)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    assert lib.ra_debug_build() == flag


def test_product_build_is_neither(ralib):
    from ring_chunked_attention_gb300 import build as rab

    prod = ctypes.CDLL(rab.LIB)
    assert prod.ra_debug_build() == 0
    assert ralib.ra_status_string(ralib.RA_ERR_BOUNDS) == "RA_ERR_BOUNDS"
    buf = (ctypes.c_ulonglong * 32)()
    prod.ra_trace_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]
    assert prod.ra_trace_read(buf, 1) == ralib.RA_ERR_UNSUPPORTED
