"""GPU parity of ra_merge_partials against the oracle's merge, and of the
composition fwd -> merge on disjoint key sets."""
import numpy as np
import pytest
import torch

from tests.parity import MAX_ABS, MEAN_ABS, assert_parity, compare

pytestmark = pytest.mark.gpu


def _partials(n, B, S, H, D, seed, empty_frac=0.1, all_empty_rows=3):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(n, B, S, H, D, generator=g)
    lse = torch.randn(n, B, H, S, generator=g) * 4.0
    drop = torch.rand(n, B, H, S, generator=g) < empty_frac
    lse[drop] = -float("inf")
    lse[:, 0, 0, :all_empty_rows] = -float("inf")  # rows with no key at all
    return o, lse


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [
    (1, 1, 128, 1, 64), (3, 2, 96, 4, 128), (8, 1, 200, 3, 64),
    (33, 2, 37, 5, 64),    # many partials: short position tiles, a ragged last tile
    (8, 1, 1000, 32, 8),   # one 16-byte vector per row
    (2, 1, 3, 4500, 8),    # n*H past the shared-memory tile budget: the per-row kernel
])
def test_merge_parity(ralib, cuda_ok, oracle_mod, dtype, shape):
    n, B, S, H, D = shape
    o, lse = _partials(n, B, S, H, D, seed=sum(shape))
    o_in = o.to(dtype)
    out, lse_out = ralib.ra_merge_partials(o_in.cuda().contiguous(), lse.cuda().contiguous())
    torch.cuda.synchronize()
    o_ref, l_ref = oracle_mod.merge(o_in.double().numpy(), lse.double().numpy())
    got = out.double().cpu().numpy()
    # out is bf16: where |out| >= 4 one half-ulp (2^-6) exceeds the max-abs gate, so
    # an element equal to the correctly rounded oracle value passes as in the
    # forward's parity checks (tests/parity.py)
    assert_parity(compare(out, None, o_ref, None), f"merge {shape} {dtype}")
    lg = lse_out.double().cpu().numpy()
    fin = np.isfinite(l_ref)
    assert (np.isneginf(lg) == np.isneginf(l_ref)).all()
    assert (np.abs(lg[fin] - l_ref[fin]) <= 1e-5 * np.maximum(1, np.abs(l_ref[fin]))).all()
    assert (got[0, :3, 0] == 0).all()


def test_merge_single_partial_is_identity(ralib, cuda_ok):
    o, lse = _partials(1, 1, 256, 2, 128, seed=5, empty_frac=0.0, all_empty_rows=0)
    ob = o.bfloat16()
    out, l2 = ralib.ra_merge_partials(ob.cuda(), lse.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), ob[0])
    assert torch.allclose(l2.cpu(), lse[0], rtol=0, atol=1e-6)


def test_fwd_then_merge_of_two_key_halves(ralib, cuda_ok, oracle_mod):
    """Non-causal attention over 2N keys = merge of attention over the first N
    and the last N keys.  Each half is computed by ra_fwd on a problem whose
    query rows are repeated to the key length, so the kernel's square shape
    requirement holds."""
    from ring_chunked_attention_gb300.inputs import Workload, make_inputs

    w = Workload("m", 1, 2, 2, 512, 128, 2, False)
    q, k, v = make_inputs(w, seed=31)
    N = w.S // 2
    qd = q.cuda()
    parts_o, parts_l = [], []
    for half in (slice(0, N), slice(N, 2 * N)):
        kk = torch.cat([k[:, half], k[:, half]], 1).cuda().contiguous()  # keys duplicated: weights unchanged
        vv = torch.cat([v[:, half], v[:, half]], 1).cuda().contiguous()
        o_h, l_h = ralib.ra_fwd(qd, kk, vv, P=1, causal=False)
        parts_o.append(o_h)
        parts_l.append(l_h - float(np.log(2.0)))  # duplicating every key doubles the sum
    out, lse = ralib.ra_merge_partials(torch.stack(parts_o).contiguous(), torch.stack(parts_l).contiguous())
    torch.cuda.synchronize()
    o_ref, l_ref = oracle_mod.attn_direct(q, k, v, False, w.scale)
    err = np.abs(out.double().cpu().numpy() - o_ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
    assert np.abs(lse.double().cpu().numpy() - l_ref).max() <= 1e-3 * max(1, np.abs(l_ref).max())
