"""GPU parity of ra_bwd (dq, dk, dv) against the fp64 oracle's gradients.

Tolerance, derived from the arithmetic (the pages state none for gradients):
every gradient element is a sum of products in which one factor was rounded
to bf16 on the way (p for dv, ds for dq and dk: relative error <= 2^-9 each),
accumulated in fp32, and the result is rounded to bf16 once more (<= 2^-9).
Errors of the rounded factors are unbiased, so on average they stay well
under one bf16 half-ulp of the gradient's scale; the gate is

    max |g - g_ref|  <= 2^-6 * max |g_ref|    (1.6 % of the tensor's largest entry)
    mean|g - g_ref|  <= 2^-8 * mean|g_ref|    (0.4 % of its mean magnitude)

per gradient tensor.

ra_bwd takes delta_s = <dout_s, out_s> on the forward output it is given
(bf16).  On near-one-hot rows ds = p (dp - delta) cancels almost completely,
so the 2^-9 rounding of out moves ds by far more than the gate above; the
oracle therefore takes delta from the same bf16 output (its own forward,
rounded), and the parity cases hand both sides the oracle's bf16 out and
fp32 lse.  End-to-end cases (ra_fwd's own out and lse fed to ra_bwd) compare
against the oracle on bf16(oracle out), which differs from ra_fwd's out only
where that rounds the other way.  Small cases compare every element with the
oracle's full gradients; the full-size workloads compare dq on a
deterministic row sample and check two exact identities of dk and dv that
hold at any size: sum over keys of dk = 0 (the rows of the softmax Jacobian
sum to zero) and sum over keys of dv = sum over the group's rows of dout (the
weights of a row sum to one), within the rounding of the bf16 outputs.
"""
import numpy as np
import pytest
import torch

from ring_chunked_attention_gb300.inputs import WORKLOADS, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

MAX_REL = 2.0 ** -6
MEAN_REL = 2.0 ** -8


def _dout(shape, seed=101):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).bfloat16()


def _fwd_bwd(ralib, q, k, v, do, w: Workload, scale=None, P=None):
    scale = w.scale if scale is None else scale
    P = w.P if P is None else P
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = ralib.ra_fwd(qd, kd, vd, P=P, causal=w.causal, scale=scale)
    dq, dk, dv = ralib.ra_bwd(qd, kd, vd, out, lse, dod, P=P, causal=w.causal, scale=scale)
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == 0
    return dq, dk, dv


def _oracle_fwd(oracle_mod, q, k, v, w: Workload, scale=None):
    """The oracle's forward, rounded the way ra_fwd returns it."""
    out, lse = oracle_mod.attn_direct(q, k, v, w.causal, w.scale if scale is None else scale)
    return torch.tensor(out).bfloat16(), torch.tensor(lse).float()


def _bwd_given(ralib, q, k, v, do, out, lse, w: Workload):
    """ra_bwd on the given (oracle) forward output and lse."""
    dq, dk, dv = ralib.ra_bwd(q.cuda(), k.cuda(), v.cuda(), out.cuda(), lse.cuda(), do.cuda(),
                              P=w.P, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == 0
    return dq, dk, dv


def _stats(got, ref):
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    err = np.abs(g - ref)
    return {"max_err": float(err.max()), "mean_err": float(err.mean()),
            "max_ref": float(np.abs(ref).max()), "mean_ref": float(np.abs(ref).mean()),
            "finite": bool(np.isfinite(g).all())}


def assert_grad(got, ref, what):
    st = _stats(got, ref)
    print(what, {k: (round(v, 6) if isinstance(v, float) else v) for k, v in st.items()})
    assert st["finite"], f"{what}: non-finite"
    assert st["max_err"] <= MAX_REL * st["max_ref"], f"{what}: {st}"
    assert st["mean_err"] <= MEAN_REL * st["mean_ref"], f"{what}: {st}"


SMALL = [
    # name, B, H, Hkv, S, D, P, causal
    ("tiny_noncausal_d64", 1, 2, 2, 256, 64, 2, False),
    ("gqa_causal_d128", 1, 4, 2, 512, 128, 2, True),
    ("mha_noncausal_d128", 2, 2, 2, 384, 128, 3, False),
    ("gqa_causal_d64_manychunks", 1, 8, 2, 1024, 64, 8, True),
    ("causal_d128_p1", 1, 2, 1, 768, 128, 1, True),
    ("single_tile", 1, 1, 1, 128, 128, 1, True),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_parity_all_elements(ralib, cuda_ok, oracle_mod, case):
    name, B, H, Hkv, S, D, P, causal = case
    w = Workload(name, B, H, Hkv, S, D, P, causal)
    q, k, v = make_inputs(w, seed=7)
    do = _dout(q.shape)
    out, lse = _oracle_fwd(oracle_mod, q, k, v, w)
    dq, dk, dv = _bwd_given(ralib, q, k, v, do, out, lse, w)
    rq, rk, rv = oracle_mod.attn_bwd(q, k, v, do, causal, w.scale, out=out)
    assert_grad(dq, rq, name + " dq")
    assert_grad(dk, rk, name + " dk")
    assert_grad(dv, rv, name + " dv")


@pytest.mark.parametrize("sigma", [3.0, 6.0])
def test_peaked_softmax(ralib, cuda_ok, oracle_mod, sigma):
    w = Workload("peak", 1, 2, 2, 512, 128, 4, True, sigma_qk=sigma)
    q, k, v = make_inputs(w, seed=23)
    do = _dout(q.shape, 24)
    out, lse = _oracle_fwd(oracle_mod, q, k, v, w)
    dq, dk, dv = _bwd_given(ralib, q, k, v, do, out, lse, w)
    rq, rk, rv = oracle_mod.attn_bwd(q, k, v, do, True, w.scale, out=out)
    assert_grad(dq, rq, f"peak{sigma} dq")
    assert_grad(dk, rk, f"peak{sigma} dk")
    assert_grad(dv, rv, f"peak{sigma} dv")


@pytest.mark.parametrize("case", [SMALL[1], SMALL[3]], ids=[SMALL[1][0], SMALL[3][0]])
def test_end_to_end_against_exact_gradient(ralib, cuda_ok, oracle_mod, case):
    """ra_fwd -> ra_bwd against the exact gradient (delta without rounding):
    on unpeaked rows the rounding of out stays inside the gate."""
    name, B, H, Hkv, S, D, P, causal = case
    w = Workload(name, B, H, Hkv, S, D, P, causal)
    q, k, v = make_inputs(w, seed=7)
    do = _dout(q.shape)
    dq, dk, dv = _fwd_bwd(ralib, q, k, v, do, w)
    rq, rk, rv = oracle_mod.attn_bwd(q, k, v, do, causal, w.scale)
    assert_grad(dq, rq, name + " e2e dq")
    assert_grad(dk, rk, name + " e2e dk")
    assert_grad(dv, rv, name + " e2e dv")


def _identities(dk, dv, do, w: Workload, what):
    """sum_t dk_t = 0 and sum_t dv_t = sum of dout over the group's rows, per
    (b, KV head, d).  Each side carries the bf16 rounding of S gradient rows,
    so the bound scales with the root-sum-square of the summed entries."""
    G = w.H // w.Hkv
    dkd, dvd = dk.double(), dv.double()
    rss_k = dkd.pow(2).sum(1).sqrt()
    assert (dkd.sum(1).abs() <= 16 * 2.0 ** -9 * rss_k + 1e-6).all(), what + " sum_t dk"
    ref_v = do.cuda().double().reshape(w.B, w.S, w.Hkv, G, w.D).sum((1, 3))
    rss_v = dvd.pow(2).sum(1).sqrt()
    err_v = (dvd.sum(1) - ref_v).abs()
    assert (err_v <= 16 * 2.0 ** -9 * rss_v + 1e-3 * ref_v.abs() + 1e-4).all(), (
        what + f" sum_t dv (max err {err_v.max().item():.3e})")


SAMPLING = {"gqa_s16384": 2048, "long_s65536": 8192, "d64_s32768": 4096}


def test_full_size_causal_s4096(ralib, cuda_ok, oracle_mod):
    w = WORKLOADS["causal_s4096"]
    q, k, v = make_inputs(w)
    do = _dout(q.shape)
    dq, dk, dv = _fwd_bwd(ralib, q, k, v, do, w)
    out, _ = _oracle_fwd(oracle_mod, q, k, v, w)
    rq, rk, rv = oracle_mod.attn_bwd(q, k, v, do, w.causal, w.scale, out=out)
    assert_grad(dq, rq, "s4096 dq")
    assert_grad(dk, rk, "s4096 dk")
    assert_grad(dv, rv, "s4096 dv")


@pytest.mark.parametrize("name", list(SAMPLING))
def test_full_size_sampled_dq_and_identities(ralib, cuda_ok, oracle_mod, name):
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    do = _dout(q.shape)
    dq, dk, dv = _fwd_bwd(ralib, q, k, v, do, w)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    rows = sample_rows(w, n_random=4, every=SAMPLING[name]).numpy()
    o_rows, _ = oracle_mod.attn_direct(q, k, v, w.causal, w.scale, rows=rows)
    ref = oracle_mod.attn_bwd_dq(q, k, v, do, w.causal, w.scale, rows,
                                 out_rows=torch.tensor(o_rows).bfloat16())
    s, h, b = rows % w.S, (rows // w.S) % w.H, rows // (w.S * w.H)
    got = dq.double().cpu().numpy()[b, s, h]
    assert_grad(got, ref, name + " dq rows")
    _identities(dk, dv, do, w, name)


# ---------------------------------------------------------------- metamorphic
def test_deterministic(ralib, cuda_ok):
    w = Workload("det", 1, 8, 2, 2048, 128, 4, True)
    q, k, v = make_inputs(w, seed=3)
    do = _dout(q.shape)
    a = _fwd_bwd(ralib, q, k, v, do, w)
    b = _fwd_bwd(ralib, q, k, v, do, w)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_p_changes_only_dq_rounding(ralib, cuda_ok):
    """dk/dv never depend on P (their query order is fixed); dq only through
    the summation order of the ring."""
    w = Workload("pinv", 1, 4, 2, 2048, 128, 1, True)
    q, k, v = make_inputs(w, seed=9)
    do = _dout(q.shape)
    base = _fwd_bwd(ralib, q, k, v, do, w, P=1)
    for P in (2, 4, 16):
        dq, dk, dv = _fwd_bwd(ralib, q, k, v, do, w, P=P)
        ref = base[0].double()
        assert (dq.double() - ref).abs().max().item() <= MAX_REL * ref.abs().max().item()
        # the forward output differs in rounding across P, so dk/dv may too;
        # they stay within the gradient tolerance of the P=1 result
        for got, r in ((dk, base[1]), (dv, base[2])):
            r = r.double()
            assert (got.double() - r).abs().max().item() <= MAX_REL * r.abs().max().item()


def test_gqa_equals_mha_on_repeated_kv(ralib, cuda_ok):
    w = Workload("gqa", 1, 8, 2, 1024, 128, 4, True)
    q, k, v = make_inputs(w, seed=13)
    do = _dout(q.shape)
    dq1, dk1, dv1 = _fwd_bwd(ralib, q, k, v, do, w)
    G = w.H // w.Hkv
    w2 = w.with_(Hkv=w.H)
    dq2, dk2, dv2 = _fwd_bwd(ralib, q, k.repeat_interleave(G, 2).contiguous(),
                             v.repeat_interleave(G, 2).contiguous(), do, w2)
    assert (dq1.float() - dq2.float()).abs().max().item() <= MAX_REL * dq2.float().abs().max().item()
    dk2s = dk2.double().reshape(1, w.S, w.Hkv, G, w.D).sum(3)
    dv2s = dv2.double().reshape(1, w.S, w.Hkv, G, w.D).sum(3)
    assert (dk1.double() - dk2s).abs().max().item() <= MAX_REL * dk2s.abs().max().item()
    assert (dv1.double() - dv2s).abs().max().item() <= MAX_REL * dv2s.abs().max().item()


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_closed_form(ralib, cuda_ok, causal):
    w = Workload("uni", 1, 4, 2, 512, 64, 2, causal)
    q, k, v = make_inputs(w, seed=17)
    do = _dout(q.shape)
    dq, dk, dv = _fwd_bwd(ralib, q, k, v, do, w, scale=0.0)
    assert not dq.any() and not dk.any()
    S, G = w.S, w.H // w.Hkv
    cnt = np.arange(1, S + 1, dtype=np.float64) if causal else np.full(S, float(S))
    grp = (do.double().numpy() / cnt[None, :, None, None]).reshape(1, S, w.Hkv, G, w.D).sum(3)
    if causal:
        ref = np.flip(np.cumsum(np.flip(grp, 1), 1), 1)
    else:
        ref = np.broadcast_to(grp.sum(1, keepdims=True), grp.shape)
    assert_grad(dv, ref, f"uniform dv causal={causal}")


def test_workspace_is_caller_owned_and_reusable(ralib, cuda_ok):
    w = Workload("ws", 1, 4, 2, 512, 128, 2, True)
    q, k, v = make_inputs(w, seed=31)
    do = _dout(q.shape)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = ralib.ra_fwd(qd, kd, vd, P=w.P, causal=True)
    ws = torch.full((ralib.ra_bwd_workspace_bytes(1, 4, 512),), 0x7F, dtype=torch.uint8,
                    device="cuda")
    r1 = ralib.ra_bwd(qd, kd, vd, out, lse, dod, P=w.P, causal=True, workspace=ws)
    r2 = ralib.ra_bwd(qd, kd, vd, out, lse, dod, P=w.P, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(r1, r2):
        assert torch.equal(x, y)
    with pytest.raises(ralib.RaError):
        ralib.ra_bwd(qd, kd, vd, out, lse, dod, P=w.P, causal=True, workspace=ws[:-16])


def test_cuda_graph_capture_and_replay(ralib, cuda_ok):
    """ra_bwd (three kernels) recorded into a CUDA graph replays to the eager
    gradients: its launches make no attribute calls once the kernels are
    prepared."""
    w = Workload("graph", 1, 8, 2, 1024, 128, 4, True)
    q, k, v = (t.cuda() for t in make_inputs(w, seed=79))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(80)).bfloat16().cuda()
    out, lse = ralib.ra_fwd(q, k, v, P=w.P, causal=True)
    ref = ralib.ra_bwd(q, k, v, out, lse, do, P=w.P, causal=True)
    dq, dk, dv = (torch.empty_like(t) for t in ref)
    ws = torch.empty(ralib.ra_bwd_workspace_bytes(w.B, w.H, w.S), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ralib.ra_bwd(q, k, v, out, lse, do, P=w.P, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ralib.ra_bwd(q, k, v, out, lse, do, P=w.P, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
    for _ in range(3):
        for t in (dq, dk, dv):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for got, r in zip((dq, dk, dv), ref):
            assert torch.equal(got, r)
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
