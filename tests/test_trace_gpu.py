"""The traced build (RA_TRACE; libringattn_trace.so): per-role cycle counters
of the forward kernel.  In a process of its own (the binding picks the library
at import, from the RA_TRACE environment variable) a paired-item launch and a
single-tile launch run with the traced library; their outputs must be the
product library's bits, and their counters must add up: the MMA warp's step count is the launch's number of
key/value steps, every CTA that ran reports, and each per-step share is a
part of the step."""
import os
import subprocess
import sys

import pytest
import torch

from ring_chunked_attention_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHILD = """
import sys, torch
sys.path.insert(0, {root!r})
import ring_chunked_attention_gb300 as ra
from ring_chunked_attention_gb300.inputs import Workload, make_inputs
from ring_chunked_attention_gb300.trace import summarize
assert ra.ra_trace_build()
w = Workload("tr", 1, 8, 2, 2048, 128, 4, True)
q, k, v = (t.cuda() for t in make_inputs(w, seed=71))
ra.ra_set_item_pairing({pairing})
out, lse = ra.ra_fwd(q, k, v, P=w.P, causal=w.causal)
torch.cuda.synchronize()
st = ra.ra_get_last_device_status()
c = ra.ra_trace_read(152)
torch.save(dict(out=out.cpu(), lse=lse.cpu(), status=st, counters=c, summary=summarize(c)), {path!r})
"""


# (pairing, key/value steps, items) of the launch: paired items are 4
# (b, head pair) groups x query tiles 0..15, each visiting key tiles 0..qt,
# 4 * (1 + 2 + ... + 16) = 544 steps over 64 items; single-tile items are
# 8 heads x the same 16 tiles, 1088 steps over 128 items
CASES = [(1, 544, 64), (2, 1088, 128)]


@pytest.mark.parametrize("pairing,steps,items", CASES, ids=["paired", "single"])
def test_traced_build_counts_and_changes_nothing(ralib, cuda_ok, tmp_path, pairing, steps, items):
    from ring_chunked_attention_gb300 import build as rab

    rab.build(trace=True)
    path = str(tmp_path / "trace.pt")
    env = dict(os.environ, RA_TRACE="1", RA_DEBUG="0")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, path=path, pairing=pairing)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = torch.load(path)
    assert res["status"] == ralib.RA_OK
    w = Workload("tr", 1, 8, 2, 2048, 128, 4, True)
    q, k, v = (t.cuda() for t in make_inputs(w, seed=71))
    ralib.ra_set_item_pairing(pairing)
    try:
        out, lse = ralib.ra_fwd(q, k, v, P=w.P, causal=w.causal)
    finally:
        ralib.ra_set_item_pairing(0)
    assert torch.equal(out.cpu(), res["out"]) and torch.equal(lse.cpu(), res["lse"])
    c = res["counters"]
    assert int(c[:, 4].sum()) == steps
    assert int(c[:, 25].sum()) == items
    ran = c[:, 5] > 0
    assert int(ran.sum()) == items               # one CTA per item (fewer items than SMs)
    assert bool((c[:, 8 + 3].sum() == steps))    # slot 0 saw every step
    s = res["summary"]
    assert s["cycles per step"] > 0
    for key in ("P waits", "PV issue", "V waits", "S issue"):
        assert 0 <= s[f"MMA warp: {key} per step"] <= s["cycles per step"]
