"""ra_bwd_static: the backward on the library's fixed device scratch (no
workspace argument, no allocation in the call).  Collected last.

Checked against the workspace entry point ra_bwd on two consecutive calls
with different inputs: each result must equal ra_bwd's bit for bit (the same
kernels in the same order read the scratch, so nothing from the first call
may leak into the second), and the device's free memory must not change
across the two calls.
"""
import ctypes

import pytest
import torch

from ring_chunked_attention_gb300.inputs import Workload, make_inputs

MAX_ROWS = 1 << 21  # query rows B*H*S the static scratch holds


def test_static_entry_rejects_oversize_before_launch(ralib):
    lib = ralib._load()
    p = 0x100000  # fake, 16-byte aligned: validation must reject before any CUDA call
    H, S = 33, 65536  # 33 * 65536 = 2,162,688 > 2^21 rows
    assert H * S > MAX_ROWS
    rc = lib.ra_bwd_static(p, p, p, p, p, p, p, p, p, 1, H, 1, S, 128, 1, 1, 0.1, None)
    assert rc == 2  # RA_ERR_UNSUPPORTED
    assert lib.ra_bwd_static(0, p, p, p, p, p, p, p, p, 1, 4, 2, 256, 128, 2, 1, 0.1, None) == 1


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_on_consecutive_calls(ralib, cuda_ok):
    w = Workload("noalloc", 1, 8, 2, 1024, 128, 4, True)
    cases = []
    for seed in (41, 42):
        q, k, v = (t.cuda() for t in make_inputs(w, seed=seed))
        g = torch.Generator().manual_seed(seed + 100)
        do = torch.randn(q.shape, generator=g).bfloat16().cuda()
        out, lse = ralib.ra_fwd(q, k, v, P=w.P, causal=True)
        ref = ralib.ra_bwd(q, k, v, out, lse, do, P=w.P, causal=True)
        got = tuple(torch.empty_like(t) for t in (q, k, v))
        cases.append((q, k, v, out, lse, do, ref, got))
    torch.cuda.synchronize()
    c = cases[0]
    ralib.ra_bwd_static(*c[:6], *c[7], P=w.P, causal=True)  # warm: kernels already loaded
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for q, k, v, out, lse, do, ref, got in cases:      # two consecutive calls
        ralib.ra_bwd_static(q, k, v, out, lse, do, *got, P=w.P, causal=True)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert ralib.ra_get_last_device_status() == 0
    assert free1 == free0
    for q, k, v, out, lse, do, ref, got in cases:
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


@pytest.mark.gpu
def test_static_scratch_at_its_largest_accepted_size(ralib, cuda_ok):
    """B*H*S == 2^21 rows exactly: the second half of the scratch (-delta) then
    ends at the last byte of the array.  The result must equal ra_bwd's with a
    workspace bit for bit."""
    w = Workload("noalloc_max", 1, 32, 8, 65536, 64, 16, True)
    assert w.B * w.H * w.S == MAX_ROWS
    q, k, v = (t.cuda() for t in make_inputs(w, seed=44))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(144)).bfloat16().cuda()
    out, lse = ralib.ra_fwd(q, k, v, P=w.P, causal=True)
    ref = ralib.ra_bwd(q, k, v, out, lse, do, P=w.P, causal=True)
    got = tuple(torch.empty_like(t) for t in (q, k, v))
    ralib.ra_bwd_static(q, k, v, out, lse, do, *got, P=w.P, causal=True)
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == 0
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
