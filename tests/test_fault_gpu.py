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
