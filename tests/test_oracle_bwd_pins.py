"""Pins of the oracle's backward pass (``ora_attn_bwd``, ``ora_attn_bwd_dq``)
against things other than itself.

The pages describe no backward pass; the oracle writes out the derivative of
the attention definition.  What fixes that derivative independently:

* central finite differences of an independent fp64 forward (numpy einsum of
  the definition) -- the derivative itself, coordinate by coordinate;
* torch autograd in fp64 through a second, independently written forward;
* closed forms: ``scale = 0`` makes every row a uniform average, so dq = dk = 0
  and dv_t = sum over the rows that see key t of dout_s / (#keys of row s);
  a causal row 0 sees one key, so its dq is 0;
* invariants at any size: the rows of the softmax Jacobian sum to zero, so
  sum_t dk_t = 0 for every (b, KV head); the weights of a row sum to one, so
  sum_t dv_t = sum of dout over the group's rows;
* GQA equals MHA on repeated K/V with dk/dv summed over the group;
* the row-sampled dq equals the full dq;
* taking delta from a given rounded output shifts dq and dk by closed forms
  in the shift of delta and leaves dv bit-identical.
"""
import numpy as np
import pytest
import torch

from ring_chunked_attention_gb300.inputs import Workload, make_inputs


def _dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).bfloat16()


def _np(x):
    return x.double().numpy()


def _fwd_einsum(q, k, v, causal, scale):
    """The definition in fp64 numpy (independent of ora.c)."""
    B, S, H, D = q.shape
    G = H // k.shape[2]
    kk, vv = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    x = scale * np.einsum("bshd,bthd->bhst", q, kk)
    if causal:
        x = np.where(np.triu(np.ones((S, S), bool), 1), -np.inf, x)
    e = np.exp(x - x.max(-1, keepdims=True))
    return np.einsum("bhst,bthd->bshd", e / e.sum(-1, keepdims=True), vv)


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences_of_the_definition(oracle_mod, causal):
    w = Workload("fd", 1, 4, 2, 6, 4, 1, causal)
    q, k, v = make_inputs(w, seed=3)
    do = _dout(q.shape, 4)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, causal, w.scale)
    args = [_np(q), _np(k), _np(v)]
    dn = _np(do)

    def loss(a):
        return float((_fwd_einsum(*a, causal, w.scale) * dn).sum())

    eps = 1e-6
    for which, grad in enumerate((dq, dk, dv)):
        fd = np.empty_like(grad)
        for idx in np.ndindex(grad.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd[idx] = (loss(plus) - loss(minus)) / (2 * eps)
        np.testing.assert_allclose(grad, fd, atol=2e-7, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_torch_autograd_fp64(oracle_mod, causal):
    w = Workload("ag", 2, 4, 2, 48, 16, 1, causal)
    q, k, v = make_inputs(w, seed=5)
    do = _dout(q.shape, 6)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, causal, w.scale)

    qt, kt, vt = (x.double().requires_grad_(True) for x in (q, k, v))
    G = w.H // w.Hkv
    kr, vr = kt.repeat_interleave(G, 2), vt.repeat_interleave(G, 2)
    x = torch.einsum("bshd,bthd->bhst", qt, kr) * w.scale
    if causal:
        x = x.masked_fill(torch.ones(w.S, w.S, dtype=torch.bool).triu(1), float("-inf"))
    out = torch.einsum("bhst,bthd->bshd", torch.softmax(x, -1), vr)
    (out * do.double()).sum().backward()
    for got, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        np.testing.assert_allclose(got, ref.numpy(), atol=1e-11, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_closed_form(oracle_mod, causal):
    w = Workload("u", 2, 4, 2, 40, 8, 1, causal)
    q, k, v = make_inputs(w, seed=7)
    do = _dout(q.shape, 8)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, causal, 0.0)
    assert not dq.any() and not dk.any()
    S, G = w.S, w.H // w.Hkv
    cnt = np.arange(1, S + 1, dtype=np.float64) if causal else np.full(S, float(S))
    wdo = _np(do) / cnt[None, :, None, None]             # dout_s / n_s
    grp = wdo.reshape(w.B, S, w.Hkv, G, w.D).sum(3)      # summed over the group's heads
    if causal:   # key t is seen by rows s >= t: reverse cumulative sum
        ref = np.flip(np.cumsum(np.flip(grp, 1), 1), 1)
    else:        # every row sees every key
        ref = np.broadcast_to(grp.sum(1, keepdims=True), grp.shape)
    np.testing.assert_allclose(dv, ref, atol=1e-12, rtol=0)


def test_invariants_and_single_key_row(oracle_mod):
    w = Workload("inv", 2, 6, 2, 96, 16, 1, True, sigma_qk=2.0)
    q, k, v = make_inputs(w, seed=9)
    do = _dout(q.shape, 10)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, True, w.scale)
    G = w.H // w.Hkv
    # sum_t ds_st = 0 for every row, hence sum_t dk_t = 0
    assert np.abs(dk.sum(1)).max() < 1e-10 * max(1.0, np.abs(dk).max())
    # rows of p sum to one, hence sum_t dv_t = sum_s dout_s over the group
    ref = _np(do).reshape(w.B, w.S, w.Hkv, G, w.D).sum((1, 3))
    np.testing.assert_allclose(dv.sum(1), ref, atol=1e-10, rtol=0)
    # causal row 0 attends to one key with weight 1: no gradient reaches q
    assert not dq[:, 0].any()
    assert np.abs(dq[:, 1:]).max() > 1e-3


def test_gqa_equals_mha_on_repeated_kv(oracle_mod):
    w = Workload("g", 1, 8, 2, 64, 16, 1, True)
    q, k, v = make_inputs(w, seed=11)
    do = _dout(q.shape, 12)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, True, w.scale)
    G = w.H // w.Hkv
    dq2, dk2, dv2 = oracle_mod.attn_bwd(q, k.repeat_interleave(G, 2), v.repeat_interleave(G, 2),
                                        do, True, w.scale)
    np.testing.assert_allclose(dq, dq2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(dk, dk2.reshape(1, w.S, w.Hkv, G, w.D).sum(3), atol=1e-12, rtol=0)
    np.testing.assert_allclose(dv, dv2.reshape(1, w.S, w.Hkv, G, w.D).sum(3), atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_dq_rows_equal_full(oracle_mod, causal):
    w = Workload("r", 2, 4, 1, 80, 8, 1, causal)
    q, k, v = make_inputs(w, seed=13)
    do = _dout(q.shape, 14)
    dq, _, _ = oracle_mod.attn_bwd(q, k, v, do, causal, w.scale)
    rows = np.array([0, 1, 79, 80 + 40, 3 * 80 + 5, 7 * 80 + 79], dtype=np.int64)
    got = oracle_mod.attn_bwd_dq(q, k, v, do, causal, w.scale, rows)
    s, h, b = rows % w.S, (rows // w.S) % w.H, rows // (w.S * w.H)
    assert np.array_equal(got, dq[b, s, h])


def test_bwd_rejects_bad_shapes(oracle_mod):
    w = Workload("bad", 1, 3, 2, 16, 8, 1, True)
    q, _, _ = make_inputs(w.with_(Hkv=3), seed=1)
    k = torch.zeros(1, 16, 2, 8).bfloat16()
    with pytest.raises(ValueError):
        oracle_mod.attn_bwd(q, k, k, q, True, 0.1)


@pytest.mark.parametrize("causal", [False, True])
def test_delta_from_given_output_shifts_by_closed_form(oracle_mod, causal):
    """With delta taken from a given (rounded) output instead of exactly,
    ds_st changes by -p_st * d_s where d_s = <dout_s, out_given_s - out_s>;
    hence dq_s moves by -scale * d_s * sum_t p_st k_t, dk_t by
    -scale * sum_s p_st d_s q_s, and dv does not move at all."""
    w = Workload("od", 1, 4, 2, 64, 16, 1, causal, sigma_qk=2.0)
    q, k, v = make_inputs(w, seed=15)
    do = _dout(q.shape, 16)
    out, _, p = oracle_mod.attn_direct(q, k, v, causal, w.scale, return_weights=True)
    out_b = torch.tensor(out).bfloat16()
    e = oracle_mod.attn_bwd(q, k, v, do, causal, w.scale)
    g = oracle_mod.attn_bwd(q, k, v, do, causal, w.scale, out=out_b)
    assert np.array_equal(g[2], e[2])
    B, S, H, D, G = w.B, w.S, w.H, w.D, w.H // w.Hkv
    d = np.einsum("bshd,bshd->bhs", _np(do), _np(out_b) - out)        # [B,H,S]
    pw = p.reshape(B, H, S, S)                                          # p[b,h,s,t]
    kk, qq = np.repeat(_np(k), G, axis=2), _np(q)
    ddq = -w.scale * np.einsum("bhs,bhst,bthd->bshd", d, pw, kk)
    ddk = -w.scale * np.einsum("bhs,bhst,bshd->bthd", d, pw, qq).reshape(B, S, w.Hkv, G, D).sum(3)
    assert np.abs(d).max() > 1e-4  # the rounding does move delta
    np.testing.assert_allclose(g[0] - e[0], ddq, atol=1e-12, rtol=0)
    np.testing.assert_allclose(g[1] - e[1], ddk, atol=1e-12, rtol=0)
    # the dq-rows mode takes the same rows of the given output
    rows = np.array([0, 5, 63, 2 * 64 + 9], dtype=np.int64)
    s_, h_ = rows % S, (rows // S) % H
    got = oracle_mod.attn_bwd_dq(q, k, v, do, causal, w.scale, rows, out_rows=out_b[0, s_, h_])
    assert np.array_equal(got, g[0][0, s_, h_])
