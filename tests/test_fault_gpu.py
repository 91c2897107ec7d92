"""Failure path on the GPU without a GPU fault: the producer is told to skip
one value-tile copy, so the consumer's bounded wait runs out (50 ms limit);
the kernel records RA_ERR_TIMEOUT in the device status word, frees its
resources and exits.  The context stays usable and the next normal launch
is correct."""
import pytest
import torch

from ring_chunked_attention_gb300.inputs import Workload, make_inputs
from tests.parity import assert_parity, compare

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_context_survives(ralib, cuda_ok, oracle_mod):
    w = Workload("fault", 1, 2, 2, 256, 64, 2, False)
    q, k, v = make_inputs(w, seed=41)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    ralib.ra_debug_set_fault(50_000_000, True)
    try:
        ralib.ra_fwd(qd, kd, vd, P=w.P, causal=False)
        assert ralib.ra_get_last_device_status() == ralib.RA_ERR_TIMEOUT
    finally:
        ralib.ra_debug_set_fault(0, False)
    # status was cleared by the read; a normal launch works and is correct
    out, lse = ralib.ra_fwd(qd, kd, vd, P=w.P, causal=False)
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    o_ref, l_ref = oracle_mod.attn_direct(q, k, v, False, w.scale)
    assert_parity(compare(out, lse, o_ref, l_ref), "after fault")
    x = torch.ones(1024, device="cuda")
    assert float((x * 2).sum()) == 2048.0
    # the aborted launch left its work-item counter at zero too: the launch that
    # takes the same counter again (64 launches later) claims every item
    w2 = Workload("fault_claims", 1, 8, 2, 4096, 128, 4, True)  # more items than SMs
    q2, k2, v2 = (t.cuda() for t in make_inputs(w2, seed=61))
    o0, l0 = ralib.ra_fwd(q2, k2, v2, P=w2.P, causal=True)
    for _ in range(65):
        o, l = ralib.ra_fwd(q2, k2, v2, P=w2.P, causal=True)
        assert torch.equal(o, o0) and torch.equal(l, l0)
    assert ralib.ra_get_last_device_status() == ralib.RA_OK


@pytest.mark.parametrize("entry", ["ra_bwd", "ra_bwd_static"])
def test_backward_timeout_is_reported_and_context_survives(ralib, cuda_ok, entry):
    """The dk/dv producer skips its first output-gradient tile copy: the MMA
    thread's bounded wait runs out, RA_ERR_TIMEOUT is reported, and the next
    normal call reproduces the result of a call made before the fault."""
    w = Workload("bfault", 1, 4, 2, 512, 128, 2, True)
    q, k, v = (t.cuda() for t in make_inputs(w, seed=43))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(44)).bfloat16().cuda()
    out, lse = ralib.ra_fwd(q, k, v, P=w.P, causal=True)

    def call():
        if entry == "ra_bwd":
            return ralib.ra_bwd(q, k, v, out, lse, do, P=w.P, causal=True)
        bufs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        return ralib.ra_bwd_static(q, k, v, out, lse, do, *bufs, P=w.P, causal=True)

    ref = call()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    ralib.ra_debug_set_fault(50_000_000, True)
    try:
        call()
        assert ralib.ra_get_last_device_status() == ralib.RA_ERR_TIMEOUT
    finally:
        ralib.ra_debug_set_fault(0, False)
    got = call()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
