"""The bounds-checked flavour of the library (RA_DEBUG) builds here without a
GPU, exports the same C ABI and says that it is the checked build; the
product build says it is not.  (Its kernels run in tests/test_debug_gpu.py.)"""
import ctypes

from tests.test_capi import _declared_functions


def test_debug_flavour_builds_and_reports_itself(ralib):
    from ring_chunked_attention_gb300 import build as rab

    path = rab.build(debug=True)
    dbg = ctypes.CDLL(path)
    missing = [n for n in _declared_functions() if not hasattr(dbg, n)]
    assert not missing, f"not exported: {missing}"
    assert dbg.ra_debug_build() == 1
    assert ctypes.CDLL(ralib.library_path()).ra_debug_build() == 0
    assert ralib.ra_status_string(ralib.RA_ERR_BOUNDS) == "RA_ERR_BOUNDS"
