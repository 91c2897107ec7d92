"""GPU parity of ra_fwd against the fp64 oracle, plus metamorphic checks.

Small cases (oracle on every row) span several 128-row tiles, every work
pairing the kernel uses (two heads of one GQA group; two consecutive tiles of
one head; a single tile), causal and non-causal, D = 64 and 128, P = 1 and
P = S/128 (one tile per chunk).  The five long-context workloads run at full
size in the launch configuration the benchmark times and are checked on a
deterministic row sample (chunk boundaries of every head plus seeded random
rows).
"""
import math

import numpy as np
import pytest
import torch

from ring_chunked_attention_gb300.inputs import WORKLOADS, Workload, make_inputs, sample_rows
from tests.parity import assert_parity, compare

pytestmark = pytest.mark.gpu


def _run(ralib, q, k, v, w: Workload, **kw):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = ralib.ra_fwd(qd, kd, vd, P=w.P, causal=w.causal, scale=kw.get("scale", w.scale))
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == 0
    return out, lse


SMALL = [
    # name, B, H, Hkv, S, D, P, causal
    ("tiny_noncausal_single", 1, 2, 2, 256, 64, 2, False),
    ("heads_causal_d128", 1, 4, 1, 512, 128, 2, True),
    ("heads_noncausal_d128", 2, 4, 2, 384, 128, 3, False),
    ("qtiles_causal_d128", 2, 3, 3, 1024, 128, 4, True),
    ("qtiles_noncausal_d64", 1, 3, 3, 512, 64, 2, False),
    ("single_causal_d64_p_eq_tiles", 1, 3, 1, 640, 64, 5, True),
    ("heads_causal_d64_manychunks", 1, 8, 2, 1024, 64, 8, True),
    ("qtiles_causal_d128_p1", 1, 1, 1, 768, 128, 1, True),
]


@pytest.fixture(params=[0, 1], ids=["auto", "paired"])
def pairing(request, ralib):
    """Work-item grouping: automatic (small launches use one query tile per
    item) and forced pairing (two heads of a group, or two consecutive tiles),
    so that every grouping is checked at sizes the oracle covers in full."""
    ralib.ra_set_item_pairing(request.param)
    yield request.param
    ralib.ra_set_item_pairing(0)


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_parity_all_rows(ralib, cuda_ok, oracle_mod, case, pairing):
    name, B, H, Hkv, S, D, P, causal = case
    w = Workload(name, B, H, Hkv, S, D, P, causal)
    q, k, v = make_inputs(w, seed=7)
    out, lse = _run(ralib, q, k, v, w)
    o_ref, l_ref = oracle_mod.attn_ring(q, k, v, P, causal, w.scale)
    st = compare(out, lse, o_ref, l_ref)
    assert_parity(st, name)


def test_tiny_workload_ring_and_direct(ralib, cuda_ok, oracle_mod):
    w = WORKLOADS["tiny"]
    q, k, v = make_inputs(w)
    out, lse = _run(ralib, q, k, v, w)
    for fn in (oracle_mod.attn_direct, lambda *a: oracle_mod.attn_ring(*a[:3], w.P, *a[3:])):
        o_ref, l_ref = fn(q, k, v, w.causal, w.scale)
        assert_parity(compare(out, lse, o_ref, l_ref), "tiny")


SAMPLING = {  # every-th row, random rows per (b, h)
    "causal_s4096": None,  # full oracle
    "gqa_s16384": (2048, 8),
    "long_s65536": (8192, 8),
    "d64_s32768": (4096, 4),
}


@pytest.mark.parametrize("name", list(SAMPLING))
def test_full_size_workload_parity(ralib, cuda_ok, oracle_mod, name):
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    out, lse = _run(ralib, q, k, v, w)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    if SAMPLING[name] is None:
        o_ref, l_ref = oracle_mod.attn_direct(q, k, v, w.causal, w.scale)
        st = compare(out, lse, o_ref, l_ref)
    else:
        every, nr = SAMPLING[name]
        rows = sample_rows(w, n_random=nr, every=every).numpy()
        o_ref, l_ref = oracle_mod.attn_direct(q, k, v, w.causal, w.scale, rows=rows)
        st = compare(out, lse, o_ref, l_ref, rows=rows)
    print(name, st)
    assert_parity(st, name)


# ---------------------------------------------------------------- metamorphic
def test_deterministic(ralib, cuda_ok):
    w = Workload("det", 1, 8, 2, 2048, 128, 4, True)
    q, k, v = make_inputs(w, seed=3)
    o1, l1 = _run(ralib, q, k, v, w)
    o2, l2 = _run(ralib, q, k, v, w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("D", [64, 128])
def test_future_chunks_do_not_reach_earlier_rows(ralib, cuda_ok, D):
    w = Workload("fut", 1, 4, 2, 1024, D, 4, True)
    q, k, v = make_inputs(w, seed=5)
    o1, l1 = _run(ralib, q, k, v, w)
    g = torch.Generator().manual_seed(11)
    C = w.chunk
    i = 1
    k2, v2 = k.clone(), v.clone()
    k2[:, (i + 1) * C:] = torch.randn(k2[:, (i + 1) * C:].shape, generator=g).bfloat16()
    v2[:, (i + 1) * C:] = torch.randn(v2[:, (i + 1) * C:].shape, generator=g).bfloat16()
    o2, l2 = _run(ralib, q, k2, v2, w)
    assert torch.equal(o1[:, : (i + 1) * C], o2[:, : (i + 1) * C])
    assert torch.equal(l1[:, :, : (i + 1) * C], l2[:, :, : (i + 1) * C])
    assert not torch.equal(o1[:, (i + 1) * C:], o2[:, (i + 1) * C:])


def test_p_invariance(ralib, cuda_ok):
    base = Workload("pinv", 1, 4, 4, 2048, 128, 1, True)
    q, k, v = make_inputs(base, seed=9)
    outs = [_run(ralib, q, k, v, base.with_(P=P)) for P in (1, 2, 4, 16)]
    o0 = outs[0][0].float()
    for o, l in outs[1:]:
        assert (o.float() - o0).abs().max().item() <= 2 * 1.5e-2
        assert (l - outs[0][1]).abs().max().item() <= 1e-3 * max(1.0, outs[0][1].abs().max().item())


def test_gqa_equals_mha_on_repeated_kv(ralib, cuda_ok):
    w = Workload("gqa", 2, 8, 2, 1024, 128, 4, True)
    q, k, v = make_inputs(w, seed=13)
    o1, l1 = _run(ralib, q, k, v, w)
    rep = w.H // w.Hkv
    w2 = w.with_(Hkv=w.H)
    o2, l2 = _run(ralib, q, k.repeat_interleave(rep, 2).contiguous(),
                  v.repeat_interleave(rep, 2).contiguous(), w2)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-4 * max(1.0, l1.abs().max().item())


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_gives_mean_of_allowed_values(ralib, cuda_ok, oracle_mod, causal):
    w = Workload("uni", 1, 2, 1, 512, 64, 2, causal)
    q, k, v = make_inputs(w, seed=17)
    out, lse = _run(ralib, q, k, v, w, scale=0.0)
    vd = v.double().numpy()
    S = w.S
    if causal:
        cnt = np.arange(1, S + 1, dtype=np.float64)
        mean = np.cumsum(vd, axis=1) / cnt[None, :, None, None]
        lse_ref = np.broadcast_to(np.log(cnt), (1, w.H, S))
    else:
        mean = np.broadcast_to(vd.mean(axis=1, keepdims=True), vd.shape)
        lse_ref = np.full((1, w.H, S), math.log(S))
    exp_out = np.repeat(mean, w.H // w.Hkv, axis=2)
    st = compare(out, lse, exp_out, lse_ref)
    assert_parity(st, "uniform")


def test_lse_optional(ralib, cuda_ok):
    w = Workload("nolse", 1, 2, 2, 256, 128, 2, True)
    q, k, v = make_inputs(w, seed=19)
    o1, _ = _run(ralib, q, k, v, w)
    o2, l2 = ralib.ra_fwd(q.cuda(), k.cuda(), v.cuda(), P=w.P, causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert l2 is None and torch.equal(o1, o2)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("sigma", [3.0, 6.0])
def test_peaked_softmax_rescaling(ralib, cuda_ok, oracle_mod, D, sigma, pairing):
    """std sigma on q and k: scores with std sigma^2 (x sqrt(D) scale), so a
    row's max jumps by far more than the 2^8 rescale threshold between tiles;
    at sigma = 6 the jumps also pass the 2^30 guard of the skipped max pass,
    so warps take the exact path (max pass, O rescale, which at D = 64 also
    rescales the PV MMA's row-sum columns).  At this size automatic grouping
    gives one query tile per item (where the O rescale first waits for the
    previous PV, which runs behind the next S); forced pairing runs the
    two-tile kernel's exact path."""
    w = Workload("peak", 1, 2, 2, 1024, D, 4, True, sigma_qk=sigma)
    q, k, v = make_inputs(w, seed=23)
    out, lse = _run(ralib, q, k, v, w)
    o_ref, l_ref = oracle_mod.attn_direct(q, k, v, True, w.scale)
    assert_parity(compare(out, lse, o_ref, l_ref), f"peaked D={D} sigma={sigma}")


@pytest.mark.parametrize("D", [64, 128])
def test_late_dominant_key_takes_the_exact_path(ralib, cuda_ok, oracle_mod, D, pairing):
    """One key of chunk 0 scores about 50 (natural units, 72 in log2 units)
    above everything else for every row of chunks 1-3.  Those rows visit
    chunk 0 last in ring order, so by then their reference max is far below
    it: the speculative exps exceed the 2^30 guard and every such warp must
    take the exact path (scores streamed back from tensor memory, new
    reference, O rescaled by about 2^-72).  The output is then dominated by
    that key's value row.  Run with one query tile per item (automatic at
    this size) and with paired items."""
    w = Workload("late", 1, 2, 1, 1024, D, 4, True)
    q, k, v = make_inputs(w, seed=31)
    t = 5                                   # the planted key (chunk 0, first tile)
    amp = math.sqrt(50.0 * math.sqrt(D))    # amp^2 * scale = 50
    q = q.float()
    k = k.float()
    q[:, w.chunk:, :, 0] += amp             # rows of chunks 1..3 share a large first component
    k[:, t] = 0.0
    k[:, t, :, 0] = amp
    q, k = q.bfloat16(), k.bfloat16()
    out, lse = _run(ralib, q, k, v, w)
    o_ref, l_ref = oracle_mod.attn_direct(q, k, v, True, w.scale)
    assert_parity(compare(out, lse, o_ref, l_ref), f"late dominant key D={D}")
    # the planted key carries nearly all the weight of the rows that see it late
    late = out[0, w.chunk:].float().cpu()
    vt = v[0, t].float()                    # [Hkv=1, D], shared by both heads
    assert (late - vt).abs().max().item() < 0.05


def _claiming_workload():
    """256 single-tile items on at most 152 SMs: every CTA claims items from the
    launch's counter after its first."""
    return Workload("claims", 1, 8, 2, 4096, 128, 4, True)


def test_work_item_counters_cycle(ralib, cuda_ok):
    """Each launch takes the next of the device's 64 work-item counters and the
    kernel leaves it at zero; over more than two full cycles every launch
    must claim every item exactly once, i.e. reproduce the first output."""
    w = _claiming_workload()
    q, k, v = (t.cuda() for t in make_inputs(w, seed=47))
    o0, l0 = ralib.ra_fwd(q, k, v, P=w.P, causal=True)
    out, lse = torch.empty_like(o0), torch.empty_like(l0)
    for _ in range(130):
        ralib.ra_fwd(q, k, v, P=w.P, causal=True, out=out, lse=lse)
        torch.cuda.synchronize()
        assert torch.equal(out, o0) and torch.equal(lse, l0)
    assert ralib.ra_get_last_device_status() == ralib.RA_OK


def test_concurrent_launches_on_two_streams(ralib, cuda_ok):
    """Two launches in flight at once on different streams use different
    counters; each reproduces its own sequential result."""
    w = _claiming_workload()
    ins = [tuple(t.cuda() for t in make_inputs(w, seed=s)) for s in (53, 59)]
    refs = [ralib.ra_fwd(*x, P=w.P, causal=True) for x in ins]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [(torch.empty_like(r[0]), torch.empty_like(r[1])) for r in refs]
    for _ in range(5):
        for x, s, (o, l) in zip(ins, streams, outs):
            with torch.cuda.stream(s):
                ralib.ra_fwd(*x, P=w.P, causal=True, out=o, lse=l, stream=s)
        torch.cuda.synchronize()
        for (o, l), (ro, rl) in zip(outs, refs):
            assert torch.equal(o, ro) and torch.equal(l, rl)
    assert ralib.ra_get_last_device_status() == ralib.RA_OK


def test_cuda_graph_capture_and_replay(ralib, cuda_ok):
    """ra_fwd recorded into a CUDA graph replays to the eager result, again and
    again: the launch makes no attribute calls once its kernel is prepared, and
    the captured launch's work-item counter is back at zero after each replay
    (this workload has more items than SMs, so every replay claims items)."""
    w = _claiming_workload()
    q, k, v = (t.cuda() for t in make_inputs(w, seed=71))
    ref_o, ref_l = ralib.ra_fwd(q, k, v, P=w.P, causal=True)
    out, lse = torch.empty_like(ref_o), torch.empty_like(ref_l)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream's device
        ralib.ra_fwd(q, k, v, P=w.P, causal=True, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ralib.ra_fwd(q, k, v, P=w.P, causal=True, out=out, lse=lse)
    for _ in range(4):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    assert ralib.ra_get_last_device_status() == ralib.RA_OK


def test_graph_replays_beside_many_eager_launches(ralib, cuda_ok):
    """A launch recorded into a CUDA graph keeps one work-item counter for every
    replay, one that eager launches never take.  Replays on one stream while
    more than 64 eager launches run on another (so the eager launches cycle
    through all their counters at least once during the replays) must each
    reproduce the sequential result bit for bit."""
    w = _claiming_workload()
    ins_g = tuple(t.cuda() for t in make_inputs(w, seed=79))
    ins_e = tuple(t.cuda() for t in make_inputs(w, seed=83))
    ref_g = ralib.ra_fwd(*ins_g, P=w.P, causal=True)
    ref_e = ralib.ra_fwd(*ins_e, P=w.P, causal=True)
    out_g, lse_g = torch.empty_like(ref_g[0]), torch.empty_like(ref_g[1])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ralib.ra_fwd(*ins_g, P=w.P, causal=True, out=out_g, lse=lse_g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ralib.ra_fwd(*ins_g, P=w.P, causal=True, out=out_g, lse=lse_g)
    torch.cuda.synchronize()
    n_eager, n_replay = 70, 24
    outs_e = [(torch.zeros_like(ref_e[0]), torch.zeros_like(ref_e[1])) for _ in range(n_eager)]
    snaps = [(torch.empty_like(ref_g[0]), torch.empty_like(ref_g[1])) for _ in range(n_replay)]
    s_g, s_e = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s_g):
        for so, sl in snaps:
            out_g.zero_()
            lse_g.zero_()
            g.replay()
            so.copy_(out_g)
            sl.copy_(lse_g)
    with torch.cuda.stream(s_e):
        for o, l in outs_e:
            ralib.ra_fwd(*ins_e, P=w.P, causal=True, out=o, lse=l, stream=s_e)
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    for so, sl in snaps:
        assert torch.equal(so, ref_g[0]) and torch.equal(sl, ref_g[1])
    for o, l in outs_e:
        assert torch.equal(o, ref_e[0]) and torch.equal(l, ref_e[1])


def test_launches_after_shutdown(ralib, cuda_ok):
    """ra_shutdown drops the host caches and starts a new kernel-preparation
    epoch; the next launches prepare again and give the same result."""
    w = Workload("shut", 1, 4, 2, 512, 128, 2, True)
    q, k, v = (t.cuda() for t in make_inputs(w, seed=73))
    o1, l1 = ralib.ra_fwd(q, k, v, P=w.P, causal=True)
    ralib.ra_shutdown()
    o2, l2 = ralib.ra_fwd(q, k, v, P=w.P, causal=True)
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_binding_checks_caller_buffers(ralib, cuda_ok):
    """Caller-provided outputs must be CUDA tensors of the right shape and dtype
    on the inputs' device: the kernels write them by address."""
    w = Workload("bufs", 1, 2, 2, 256, 64, 2, True)
    q, k, v = (t.cuda() for t in make_inputs(w, seed=67))
    with pytest.raises(ValueError):
        ralib.ra_fwd(q, k, v, P=w.P, causal=True, out=torch.empty(q.shape, dtype=q.dtype))
    with pytest.raises(ValueError):
        ralib.ra_fwd(q, k, v, P=w.P, causal=True, lse=torch.empty(1, 2, 256))
    with pytest.raises(ValueError):
        ralib.ra_fwd(q, k, v, P=w.P, causal=True, out=torch.empty_like(q)[:, :128])
    with pytest.raises(ValueError):
        ralib.ra_fwd_block(q, k, v, q_pos0=0, k_pos0=0, causal=True,
                           out=torch.empty(1, 128, 2, 64, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        ralib.ra_fwd_block(q, k, v, q_pos0=0, k_pos0=0, causal=True,
                           lse=torch.empty(1, 2, 256, dtype=torch.float64, device="cuda"))
    out, lse = ralib.ra_fwd(q, k, v, P=w.P, causal=True)
    with pytest.raises(ValueError):
        ralib.ra_bwd(q, k, v, out, lse, torch.randn_like(q), P=w.P, causal=True,
                     workspace=torch.empty(1 << 16, dtype=torch.uint8))
    with pytest.raises(ValueError):
        ralib.ra_merge_partials(out[None].float(), lse[None], out=torch.empty_like(out).float())
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK


def test_stream_argument_is_used(ralib, cuda_ok, oracle_mod):
    w = Workload("stream", 1, 4, 2, 512, 128, 2, True)
    q, k, v = make_inputs(w, seed=29)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, lse = ralib.ra_fwd(qd, kd, vd, P=w.P, causal=True, stream=s)
    s.synchronize()
    o_ref, l_ref = oracle_mod.attn_direct(q, k, v, True, w.scale)
    assert_parity(compare(out, lse, o_ref, l_ref), "side stream")


@pytest.mark.parametrize("name", ["tiny", "causal_s4096", "gqa_s16384", "long_s65536",
                                  "d64_s32768", "small"])
def test_mma_orders_are_bit_identical(ralib, cuda_ok, name):
    """The four MMA issue orders run the same arithmetic in the same
    accumulation order; they differ only in how the next S product of a query
    tile is ordered after the PV product that reads the columns it rewrites
    (a tcgen05.shift between them, a commit wait, both PVs first, or nothing).
    Any ordering hazard would corrupt P and show up as a difference.  Every
    workload runs under every order twice: with paired query tiles forced (the
    pairs are where the orders differ) and with one query tile per item forced
    (those launches run their own loop, S two steps ahead in double-buffered
    columns, whatever the order).  Pairing changes which SM runs a tile, not
    its arithmetic, so all ten results are the same bits."""
    w = WORKLOADS[name] if name in WORKLOADS else Workload("small", 2, 8, 2, 2048, 128, 4, True)
    q, k, v = make_inputs(w, seed=43)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    outs = []
    try:
        for pairing in (1, 2):
            ralib.ra_set_item_pairing(pairing)
            for order in (ralib.MMA_ORDER_BRIDGED, ralib.MMA_ORDER_STRICT,
                          ralib.MMA_ORDER_GROUPED, ralib.MMA_ORDER_INORDER,
                          ralib.MMA_ORDER_BRIDGED):
                ralib.ra_set_mma_order(order)
                o, l = ralib.ra_fwd(qd, kd, vd, P=w.P, causal=w.causal)
                torch.cuda.synchronize()
                assert ralib.ra_get_last_device_status() == 0
                outs.append((o, l))
                del o, l
    finally:
        ralib.ra_set_mma_order(ralib.MMA_ORDER_BRIDGED)
        ralib.ra_set_item_pairing(0)
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_bridged_order_under_contention(ralib, cuda_ok):
    """The default order relies on tcgen05.mma -> tcgen05.shift -> tcgen05.mma
    executing in issue order; any hazard would depend on timing.  Paired and
    single-tile launches of three shapes (D = 128 and 64) run together on four
    streams, several rounds, so that CTAs of different launches share SMs and
    the copy engines and L2 are contended; every result must equal the same
    call made alone under the commit-wait order."""
    shapes = [Workload("c1", 2, 8, 2, 2048, 128, 4, True), Workload("c2", 1, 6, 3, 1536, 64, 3, True),
              Workload("c3", 1, 4, 4, 1024, 128, 2, False)]
    ins = [tuple(t.cuda() for t in make_inputs(w, seed=61 + i)) for i, w in enumerate(shapes)]
    ralib.ra_set_mma_order(ralib.MMA_ORDER_STRICT)
    try:
        refs = [ralib.ra_fwd(*x, P=w.P, causal=w.causal) for x, w in zip(ins, shapes)]
        torch.cuda.synchronize()
    finally:
        ralib.ra_set_mma_order(ralib.MMA_ORDER_BRIDGED)
    streams = [torch.cuda.Stream() for _ in range(4)]
    jobs = [(i % len(shapes), streams[i]) for i in range(4)]
    outs = [(torch.empty_like(refs[j][0]), torch.empty_like(refs[j][1])) for j, _ in jobs]
    for rnd in range(6):
        ralib.ra_set_item_pairing(rnd % 3)
        try:
            for (j, s), (o, l) in zip(jobs, outs):
                with torch.cuda.stream(s):
                    ralib.ra_fwd(*ins[j], P=shapes[j].P, causal=shapes[j].causal, out=o, lse=l,
                                 stream=s)
            torch.cuda.synchronize()
        finally:
            ralib.ra_set_item_pairing(0)
        assert ralib.ra_get_last_device_status() == ralib.RA_OK
        for (j, _), (o, l) in zip(jobs, outs):
            assert torch.equal(o, refs[j][0]) and torch.equal(l, refs[j][1]), (rnd, j)
