"""GPU parity of ra_fwd_block (one ring step) against the oracle's block, and
the ring emulated on one GPU: rank i's query chunk against every key/value
chunk in ring order, partials merged with ra_merge_partials, equals ra_fwd."""
import numpy as np
import pytest
import torch

from ring_chunked_attention_gb300.inputs import Workload, make_inputs
from tests.parity import assert_parity, compare

pytestmark = pytest.mark.gpu

CASES = [
    # name, B, H, Hkv, Sq, Sk, D, q_pos0, k_pos0, causal
    ("diag_block_heads", 1, 4, 2, 256, 256, 128, 512, 512, True),
    ("past_block_qtiles", 2, 3, 3, 512, 384, 128, 1024, 256, True),
    ("future_block_empty", 1, 2, 1, 256, 256, 64, 0, 256, True),
    ("straddling_block", 1, 2, 2, 384, 256, 128, 128, 256, True),
    ("noncausal_block", 1, 4, 4, 256, 640, 64, 0, 4096, False),
    ("single_tile_rows", 1, 3, 1, 128, 256, 128, 128, 0, True),
    ("diag_block_d64_qtiles", 1, 3, 3, 256, 384, 64, 256, 128, True),
    # more work items than SMs (run-time claims), half of them with no allowed key
    ("many_items_half_empty", 1, 8, 8, 4096, 2048, 128, 0, 2048, True),
]


@pytest.fixture(params=[0, 1], ids=["auto", "paired"])
def pairing(request, ralib):
    """Automatic work-item grouping and forced pairing of query tiles."""
    ralib.ra_set_item_pairing(request.param)
    yield request.param
    ralib.ra_set_item_pairing(0)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_block_parity(ralib, cuda_ok, oracle_mod, case, pairing):
    name, B, H, Hkv, Sq, Sk, D, qp, kp, causal = case
    g = torch.Generator().manual_seed(sum(case[1:8]))
    q = torch.randn(B, Sq, H, D, generator=g).bfloat16()
    k = torch.randn(B, Sk, Hkv, D, generator=g).bfloat16()
    v = torch.randn(B, Sk, Hkv, D, generator=g).bfloat16()
    scale = D ** -0.5
    out, lse = ralib.ra_fwd_block(q.cuda(), k.cuda(), v.cuda(), q_pos0=qp, k_pos0=kp, causal=causal)
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == 0
    o_ref, l_ref = oracle_mod.attn_block(q, k, v, qp, kp, causal, scale)
    empty = np.isneginf(l_ref)
    lg = lse.double().cpu().numpy()
    assert (np.isneginf(lg) == empty).all()
    og = out.double().cpu().numpy()
    assert (og[np.broadcast_to(empty.transpose(0, 2, 1)[..., None], og.shape)] == 0).all()
    if (~empty).any():
        l_cmp = np.where(empty, 0.0, l_ref)
        st = compare(out, torch.tensor(np.where(empty, 0.0, lg)), o_ref, l_cmp)
        assert_parity(st, name)


@pytest.mark.parametrize("causal", [True, False])
def test_ring_of_blocks_on_one_gpu_equals_ra_fwd(ralib, cuda_ok, causal):
    w = Workload("ring", 1, 8, 2, 2048, 128, 4, causal)
    q, k, v = make_inputs(w, seed=47)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    full, full_lse = ralib.ra_fwd(qd, kd, vd, P=w.P, causal=causal)
    C = w.chunk
    for i in range(w.P):  # rank i's view of the ring
        qi = qd[:, i * C:(i + 1) * C].contiguous()
        parts_o, parts_l = [], []
        for t in range(w.P):
            j = (i - t) % w.P  # block received at ring step t
            kj = kd[:, j * C:(j + 1) * C].contiguous()
            vj = vd[:, j * C:(j + 1) * C].contiguous()
            o, l = ralib.ra_fwd_block(qi, kj, vj, q_pos0=i * C, k_pos0=j * C, causal=causal)
            parts_o.append(o)
            parts_l.append(l)
        om, lm = ralib.ra_merge_partials(torch.stack(parts_o).contiguous(),
                                         torch.stack(parts_l).contiguous())
        torch.cuda.synchronize()
        ref_o = full[:, i * C:(i + 1) * C].float()
        assert (om.float() - ref_o).abs().max().item() <= 2 * 1.5e-2
        assert (om.float() - ref_o).abs().mean().item() <= 2e-3
        ref_l = full_lse[:, :, i * C:(i + 1) * C]
        assert ((lm - ref_l).abs() / ref_l.abs().clamp(min=1)).max().item() <= 1e-3
