"""The bounds-checked build (RA_DEBUG; libringattn_debug.so).

compute-sanitizer is not available, so the library has a flavour whose
kernels check every global address they compute against its buffer, set a
status bit and skip the access when it falls outside.  Two properties are
checked, each in processes of their own (the binding picks the library at
import, from the RA_DEBUG environment variable):

* on awkward small shapes, every entry point of the checked build reports no
  out-of-bounds access and returns the same bits as the product build (the
  checks change no arithmetic);
* the checks fire: with the test hook that makes the last elements of every
  buffer count as outside it, the status is RA_ERR_BOUNDS (not a timeout: a
  skipped bulk copy still completes its barrier), the hooked elements keep
  their previous contents and every other element is what an unhooked call
  writes.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRIPT = os.path.join(ROOT, "tests", "debug_checks.py")


def _run(tmp_path, debug, *flags):
    from ring_chunked_attention_gb300 import build as rab

    rab.build(debug=debug)
    path = os.path.join(str(tmp_path), f"res_{int(debug)}.pt")
    env = dict(os.environ, RA_DEBUG="1" if debug else "0")
    r = subprocess.run([sys.executable, SCRIPT, path, *flags], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return torch.load(path)


@pytest.fixture(scope="module")
def results(tmp_path_factory, cuda_ok):
    tmp = tmp_path_factory.mktemp("dbg")
    return _run(tmp, True, "--trim"), _run(tmp, False)


def test_checked_build_is_loaded(results):
    dbg, prod = results
    assert dbg["debug_build"] == 1 and prod["debug_build"] == 0


def test_no_access_outside_any_buffer_and_same_bits(results):
    import ring_chunked_attention_gb300 as ra

    dbg, prod = results
    keys = [k for k in prod if k not in ("debug_build",)]
    assert keys
    for k in keys:
        *tensors, status = dbg[k]
        *ref, ref_status = prod[k]
        assert status == ra.RA_OK, (k, status)
        assert ref_status == ra.RA_OK, (k, ref_status)
        for a, b in zip(tensors, ref):
            assert torch.equal(a, b), k


def test_the_checks_fire_and_skip_only_the_hooked_elements(results):
    import ring_chunked_attention_gb300 as ra

    t = results[0]["trim"]
    assert t["st_fwd"] == ra.RA_ERR_BOUNDS
    assert t["st_bwd"] == ra.RA_ERR_BOUNDS
    assert t["st_merge"] == ra.RA_ERR_BOUNDS
    n = t["trim"]
    for got, ref in ((t["out"], t["out0"]), (t["lse"], t["lse0"])):
        g, r = got.reshape(-1), ref.reshape(-1)
        # every store whose range reaches into the hooked tail is skipped: the
        # tail keeps the sentinel, and so may the rest of a skipped 8-element
        # vector or row; everything before that is the unhooked result
        assert bool((g[-n:].float() == t["sentinel"]).all())
        keep = g.numel() - n - 128  # a skipped row or vector reaches back at most 128 elements
        assert torch.equal(g[:keep], r[:keep])
    m = t["mout"].reshape(-1)
    assert bool((m[-n:].float() == t["sentinel"]).all())
