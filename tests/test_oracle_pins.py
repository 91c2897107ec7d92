"""Pins of the fp64 oracle against things other than itself (CPU only).

The pages print no worked attention example, so every pin comes from what the
definition of exact softmax attention fixes (mKernel overview page, table
"Die fünf verschmolzenen Kerne", row Ring Attention: the local step is
FlashAttention, fed one ring block at a time):

* hand-derived closed-form fixtures under ``tests/golden/`` (exact rationals);
* uniform scores (scale = 0 or q = 0): the output is the mean of the allowed
  value rows and lse = ln(#allowed keys);
* causal row 0 sees one key: out = v[0], lse = its score;
* two keys: the weights are a logistic function of the score gap;
* the weights of a row are positive, sum to 1, and out = weights @ v;
* future chunks never reach earlier rows (bit-identical under replacement);
* GQA equals MHA on head-repeated K/V; non-causal output is invariant under a
  joint permutation of keys and values;
* the ring fold equals the direct two-pass result for every P dividing S;
* merging partials over disjoint key sets (computed with numpy) equals the
  direct result over all keys; merge algebra on closed forms;
* brute force with ``numpy.einsum`` on tiny shapes.

A plausible slip in the oracle (dropped scale, wrong GQA index, off-by-one
causal bound, wrong log base, wrong ring fold weight, transposed operand)
fails at least one of these.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from ring_chunked_attention_gb300.inputs import WORKLOADS, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


def _rand(B, S, H, Hkv, D, seed=0, sq=1.0, sv=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, S, H, D, generator=g) * sq).to(torch.bfloat16)
    k = (torch.randn(B, S, Hkv, D, generator=g) * sq).to(torch.bfloat16)
    v = (torch.randn(B, S, Hkv, D, generator=g) * sv).to(torch.bfloat16)
    return q, k, v


def _einsum_ref(q, k, v, causal, scale):
    """Independent brute force with numpy.einsum (fp64)."""
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    B, S, H, D = qd.shape
    Hkv = kd.shape[2]
    rep = H // Hkv
    kd = np.repeat(kd, rep, axis=2)
    vd = np.repeat(vd, rep, axis=2)
    x = np.einsum("bshd,bthd->bhst", qd, kd) * scale
    if causal:
        x = np.where(np.tril(np.ones((S, S), bool))[None, None], x, -np.inf)
    m = x.max(-1, keepdims=True)
    e = np.exp(x - m)
    L = e.sum(-1, keepdims=True)
    out = np.einsum("bhst,bthd->bshd", e / L, vd)
    lse = (m + np.log(L))[..., 0]
    return out, lse


# ---------------------------------------------------------------- fixtures --
def _parse_golden(path):
    cases, cur, header = [], None, {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"causal": int(vals[0].split("=")[1])}
                cases.append(cur)
            elif cur is None:
                header[key] = vals
            else:
                cur[key] = vals
    B, H, Hkv, S, D = map(int, header["shape"])
    assert header["scale"] == ["ln2"]
    q = np.array(header["q"], float).reshape(B, S, H, D)
    k = np.array(header["k"], float).reshape(B, S, Hkv, D)
    v = np.array(header["v"], float).reshape(B, S, Hkv, D)
    for c in cases:
        c["out"] = np.array([float(Fraction(x)) for x in c["out"]]).reshape(B, S, H, D)
        c["lse"] = np.log(np.array([float(Fraction(x)) for x in c["lse_ln"]])).reshape(B, H, S)
    return q, k, v, math.log(2.0), cases


@pytest.mark.parametrize("name", ["powers_of_two.txt", "gqa_groups.txt"])
def test_golden_fixtures(oracle_mod, name):
    q, k, v, scale, cases = _parse_golden(os.path.join(GOLDEN, name))
    S = q.shape[1]
    qb, kb, vb = _bf16(q), _bf16(k), _bf16(v)
    for c in cases:
        out, lse = oracle_mod.attn_direct(qb, kb, vb, c["causal"], scale)
        np.testing.assert_allclose(out, c["out"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, c["lse"], rtol=0, atol=1e-12)
        for P in [p for p in range(1, S + 1) if S % p == 0]:
            out_r, lse_r = oracle_mod.attn_ring(qb, kb, vb, P, c["causal"], scale)
            np.testing.assert_allclose(out_r, c["out"], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse_r, c["lse"], rtol=0, atol=1e-12)


# ------------------------------------------------------------ closed forms --
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("zero", ["scale", "q"])
def test_uniform_scores_give_mean_of_v(oracle_mod, causal, zero):
    B, S, H, Hkv, D = 2, 64, 4, 2, 8
    q, k, v = _rand(B, S, H, Hkv, D, seed=3)
    scale = 0.0 if zero == "scale" else 0.7
    if zero == "q":
        q = torch.zeros_like(q)
    vd = _f64(v)
    if causal:
        cnt = np.arange(1, S + 1, dtype=np.float64)
        mean = np.cumsum(vd, axis=1) / cnt[None, :, None, None]
        lse_ref = np.broadcast_to(np.log(cnt), (B, H, S))
    else:
        mean = np.broadcast_to(vd.mean(axis=1, keepdims=True), vd.shape)
        lse_ref = np.full((B, H, S), math.log(S))
    exp_out = np.repeat(mean, H // Hkv, axis=2)
    for fn in (lambda: oracle_mod.attn_direct(q, k, v, causal, scale),
               lambda: oracle_mod.attn_ring(q, k, v, 4, causal, scale)):
        out, lse = fn()
        np.testing.assert_allclose(out, exp_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_causal_row0_is_single_key(oracle_mod):
    B, S, H, Hkv, D = 2, 32, 4, 4, 16
    q, k, v = _rand(B, S, H, Hkv, D, seed=5)
    scale = 0.3
    out, lse = oracle_mod.attn_direct(q, k, v, True, scale)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    np.testing.assert_array_equal(out[:, 0], vd[:, 0])
    dot = np.einsum("bhd,bhd->bh", qd[:, 0], kd[:, 0])
    np.testing.assert_allclose(lse[:, :, 0], scale * dot, rtol=0, atol=1e-12)


def test_two_keys_logistic(oracle_mod):
    # S=2 non-causal: weight of key 0 = 1 / (1 + e^{x1 - x0})
    q, k, v = _rand(1, 2, 3, 3, 4, seed=7)
    scale = 0.9
    out, lse = oracle_mod.attn_direct(q, k, v, False, scale)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    for s in range(2):
        for h in range(3):
            x0 = scale * float(qd[0, s, h] @ kd[0, 0, h])
            x1 = scale * float(qd[0, s, h] @ kd[0, 1, h])
            w0 = 1.0 / (1.0 + math.exp(x1 - x0))
            exp = w0 * vd[0, 0, h] + (1 - w0) * vd[0, 1, h]
            np.testing.assert_allclose(out[0, s, h], exp, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[0, h, s], max(x0, x1) + math.log1p(math.exp(-abs(x1 - x0))),
                                       rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_weights_rows_sum_to_one(oracle_mod, causal):
    B, S, H, Hkv, D = 1, 48, 2, 1, 8
    q, k, v = _rand(B, S, H, Hkv, D, seed=11, sq=2.0)
    scale = 0.5
    out, lse, w = oracle_mod.attn_direct(q, k, v, causal, scale, return_weights=True)
    w = w.reshape(B, H, S, S)
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=0, atol=1e-14)
    assert (w >= 0).all()
    if causal:
        assert (w[..., np.triu_indices(S, 1)[0], np.triu_indices(S, 1)[1]] == 0).all()
        assert (np.diagonal(w, axis1=-2, axis2=-1) > 0).all()
    # out = weights @ v
    vd = np.repeat(_f64(v), H // Hkv, axis=2)
    np.testing.assert_allclose(out, np.einsum("bhst,bthd->bshd", w, vd), rtol=0, atol=1e-12)
    # the weights are e^{x - lse}: their log-ratio equals the score gap
    qd, kd = _f64(q), np.repeat(_f64(k), H // Hkv, axis=2)
    x = scale * np.einsum("bshd,bthd->bhst", qd, kd)
    lw = np.log(np.where(w > 0, w, 1.0))
    mask = w > 0
    np.testing.assert_allclose(lw[mask], (x - lse[..., None])[mask], rtol=0, atol=1e-11)


# -------------------------------------------------------------- invariants --
@pytest.mark.parametrize("mode", ["direct", "ring"])
def test_future_chunks_contribute_nothing(oracle_mod, mode):
    B, S, H, Hkv, D, P = 1, 64, 2, 2, 8, 4
    C = S // P
    q, k, v = _rand(B, S, H, Hkv, D, seed=13)
    k2, v2 = k.clone(), v.clone()
    g = torch.Generator().manual_seed(99)
    i = 1  # rows of chunk 1; chunks 2,3 are in its future
    k2[:, (i + 1) * C:] = torch.randn(k2[:, (i + 1) * C:].shape, generator=g).to(torch.bfloat16)
    v2[:, (i + 1) * C:] = torch.randn(v2[:, (i + 1) * C:].shape, generator=g).to(torch.bfloat16)
    run = (lambda kk, vv: oracle_mod.attn_direct(q, kk, vv, True, 0.35)) if mode == "direct" else \
        (lambda kk, vv: oracle_mod.attn_ring(q, kk, vv, P, True, 0.35))
    o1, l1 = run(k, v)
    o2, l2 = run(k2, v2)
    np.testing.assert_array_equal(o1[:, : (i + 1) * C], o2[:, : (i + 1) * C])
    np.testing.assert_array_equal(l1[:, :, : (i + 1) * C], l2[:, :, : (i + 1) * C])
    assert not np.array_equal(o1[:, (i + 1) * C:], o2[:, (i + 1) * C:])


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_on_repeated_kv(oracle_mod, causal):
    B, S, H, Hkv, D = 2, 40, 6, 2, 8
    q, k, v = _rand(B, S, H, Hkv, D, seed=17)
    rep = H // Hkv
    o1, l1 = oracle_mod.attn_direct(q, k, v, causal, 0.4)
    o2, l2 = oracle_mod.attn_direct(q, k.repeat_interleave(rep, 2), v.repeat_interleave(rep, 2), causal, 0.4)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # a wrong mapping (h % Hkv) would differ from this
    o3, _ = oracle_mod.attn_direct(q, k.repeat(1, 1, rep, 1), v.repeat(1, 1, rep, 1), causal, 0.4)
    assert not np.allclose(o1, o3)


def test_noncausal_permutation_invariance(oracle_mod):
    B, S, H, Hkv, D = 1, 50, 2, 1, 16
    q, k, v = _rand(B, S, H, Hkv, D, seed=19)
    perm = torch.randperm(S, generator=torch.Generator().manual_seed(4))
    o1, l1 = oracle_mod.attn_direct(q, k, v, False, 0.25)
    o2, l2 = oracle_mod.attn_direct(q, k[:, perm], v[:, perm], False, 0.25)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [16, 24, 36])
def test_ring_fold_equals_direct_for_every_P(oracle_mod, causal, S):
    B, H, Hkv, D = 1, 4, 2, 8
    q, k, v = _rand(B, S, H, Hkv, D, seed=23, sq=3.0)  # peaked softmax
    od, ld = oracle_mod.attn_direct(q, k, v, causal, 1.0 / math.sqrt(D))
    for P in [p for p in range(1, S + 1) if S % p == 0]:
        orr, lr = oracle_mod.attn_ring(q, k, v, P, causal, 1.0 / math.sqrt(D))
        np.testing.assert_allclose(orr, od, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lr, ld, rtol=1e-12, atol=1e-12)


def test_ring_fold_on_tiny_workload_rows(oracle_mod):
    w = WORKLOADS["tiny"]
    q, k, v = make_inputs(w)
    od, ld = oracle_mod.attn_direct(q, k, v, w.causal, w.scale)
    orr, lr = oracle_mod.attn_ring(q, k, v, w.P, w.causal, w.scale)
    np.testing.assert_allclose(orr, od, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lr, ld, rtol=1e-12, atol=1e-13)
    # sampled-row interface agrees with the full run
    rows = np.array([0, 5, 127, 128, 255, 256 + 3, 511], np.int64)
    o_s, l_s = oracle_mod.attn_ring(q, k, v, w.P, w.causal, w.scale, rows=rows)
    B, S, H, D = q.shape
    for n, r in enumerate(rows):
        s, h, b = r % S, (r // S) % H, r // (S * H)
        np.testing.assert_array_equal(o_s[n], orr[b, s, h])
        assert l_s[n] == lr[b, h, s]


# -------------------------------------------------------------- brute force --
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 8, 1, 1, 4), (2, 33, 4, 2, 16), (1, 64, 3, 1, 32)])
def test_direct_matches_einsum_bruteforce(oracle_mod, causal, shape):
    B, S, H, Hkv, D = shape
    q, k, v = _rand(B, S, H, Hkv, D, seed=29, sq=1.5)
    scale = 1.0 / math.sqrt(D)
    o, l = oracle_mod.attn_direct(q, k, v, causal, scale)
    oe, le = _einsum_ref(q, k, v, causal, scale)
    np.testing.assert_allclose(o, oe, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, le, rtol=0, atol=1e-12)


# -------------------------------------------------------------------- merge --
def test_merge_of_disjoint_key_sets_equals_direct(oracle_mod):
    B, S, H, Hkv, D = 1, 30, 2, 2, 8
    q, k, v = _rand(B, S, H, Hkv, D, seed=31)
    scale = 0.4
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    sets = [np.arange(0, 7), np.arange(7, 19), np.arange(19, 30)]
    o_parts, l_parts = [], []
    for idx in sets:  # partials over a key subset, with numpy
        x = np.einsum("bshd,bthd->bhst", qd, kd[:, idx]) * scale
        m = x.max(-1, keepdims=True)
        e = np.exp(x - m)
        L = e.sum(-1, keepdims=True)
        o_parts.append(np.einsum("bhst,bthd->bshd", e / L, vd[:, idx]))
        l_parts.append((m + np.log(L))[..., 0])
    out, lse = oracle_mod.merge(np.stack(o_parts), np.stack(l_parts))
    od, ld = oracle_mod.attn_direct(q, k, v, False, scale)
    np.testing.assert_allclose(out, od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ld, rtol=0, atol=1e-12)


def test_merge_closed_forms(oracle_mod):
    rng = np.random.default_rng(0)
    B, S, H, D = 1, 3, 2, 4
    oa = rng.standard_normal((B, S, H, D))
    ob = rng.standard_normal((B, S, H, D))
    a, b = 3.0, 5.0
    la = np.full((B, H, S), math.log(a))
    lb = np.full((B, H, S), math.log(b))
    out, lse = oracle_mod.merge(np.stack([oa, ob]), np.stack([la, lb]))
    np.testing.assert_allclose(out, (a * oa + b * ob) / (a + b), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(a + b), rtol=0, atol=1e-14)
    # identical partials: same output, lse + ln 2
    out, lse = oracle_mod.merge(np.stack([oa, oa]), np.stack([la, la]))
    np.testing.assert_allclose(out, oa, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, la + math.log(2), rtol=0, atol=1e-14)
    # an empty partial adds nothing; all empty gives 0 and -inf
    ninf = np.full((B, H, S), -np.inf)
    out, lse = oracle_mod.merge(np.stack([oa, ob]), np.stack([la, ninf]))
    np.testing.assert_array_equal(out, oa)
    np.testing.assert_array_equal(lse, la)
    out, lse = oracle_mod.merge(np.stack([oa, ob]), np.stack([ninf, ninf]))
    assert (out == 0).all() and np.isneginf(lse).all()
    # n = 1 is the identity
    out, lse = oracle_mod.merge(oa[None], la[None])
    np.testing.assert_array_equal(out, oa)
    np.testing.assert_array_equal(lse, la)


def test_rejects_bad_shapes(oracle_mod):
    q, k, v = _rand(1, 10, 3, 2, 4)
    with pytest.raises(ValueError):
        oracle_mod.attn_direct(q, k, v, False, 1.0)  # H % Hkv != 0
    q, k, v = _rand(1, 10, 2, 2, 4)
    with pytest.raises(ValueError):
        oracle_mod.attn_ring(q, k, v, 3, False, 1.0)  # S % P != 0


# -------------------------------------------------------------- ring block --
@pytest.mark.parametrize("causal", [False, True])
def test_block_over_whole_sequence_is_direct(oracle_mod, causal):
    q, k, v = _rand(2, 48, 4, 2, 8, seed=37)
    od, ld = oracle_mod.attn_direct(q, k, v, causal, 0.3)
    ob, lb = oracle_mod.attn_block(q, k, v, 0, 0, causal, 0.3)
    np.testing.assert_allclose(ob, od, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lb, ld, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_ring_of_blocks_merges_to_direct(oracle_mod, causal):
    """Rank i holds query chunk i; at ring step t it receives key/value chunk
    j = (i - t) mod P and computes that block's partial; merging the P
    partials gives exact attention over all keys."""
    B, S, H, Hkv, D, P = 1, 60, 2, 1, 8, 4
    C = S // P
    q, k, v = _rand(B, S, H, Hkv, D, seed=41, sq=2.0)
    od, ld = oracle_mod.attn_direct(q, k, v, causal, 0.45)
    for i in range(P):
        qi = q[:, i * C:(i + 1) * C]
        parts = [oracle_mod.attn_block(qi, k[:, j * C:(j + 1) * C], v[:, j * C:(j + 1) * C],
                                       i * C, j * C, causal, 0.45)
                 for j in [(i - t) % P for t in range(P)]]
        om, lm = oracle_mod.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(om, od[:, i * C:(i + 1) * C], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lm, ld[:, :, i * C:(i + 1) * C], rtol=0, atol=1e-12)


def test_block_in_the_future_is_empty(oracle_mod):
    q, k, v = _rand(1, 16, 2, 2, 8, seed=43)
    ob, lb = oracle_mod.attn_block(q, k, v, 0, 16, True, 0.5)  # all keys after all queries
    assert (ob == 0).all() and np.isneginf(lb).all()
    ob, lb = oracle_mod.attn_block(q, k, v, 0, 16, False, 0.5)  # non-causal: everything allowed
    assert np.isfinite(lb).all()


def test_block_offsets_on_golden_fixture(oracle_mod):
    """Query rows 1..2 of the powers-of-two fixture, given as a block at
    position 1 against all keys at position 0, reproduce the fixture's rows."""
    q, k, v, scale, cases = _parse_golden(os.path.join(GOLDEN, "powers_of_two.txt"))
    for c in cases:
        ob, lb = oracle_mod.attn_block(_bf16(q[:, 1:]), _bf16(k), _bf16(v), 1, 0, c["causal"], scale)
        np.testing.assert_allclose(ob, c["out"][:, 1:], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lb, c["lse"][:, :, 1:], rtol=0, atol=1e-12)
