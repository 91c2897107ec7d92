"""Calls every entry point of the library the binding loads, on awkward small
shapes, and saves the outputs and device statuses to a file (torch.save).

Run by ``tests/test_debug_gpu.py`` twice: once with ``RA_DEBUG=1`` (the
bounds-checked build) and once without (the product build), each in a process
of its own; the test then compares the two files.  With ``--trim`` it also
runs the bounds-check test hook (the last elements of every buffer count as
outside it) and records what the checks left untouched.

Usage: python tests/debug_checks.py OUT_FILE [--trim]
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import ring_chunked_attention_gb300 as ra  # noqa: E402
from ring_chunked_attention_gb300.inputs import Workload, make_inputs  # noqa: E402

FWD = [  # B, H, Hkv, S, D, P, causal
    (1, 3, 1, 640, 64, 5, True),
    (2, 5, 5, 384, 128, 3, False),
    (1, 4, 2, 1024, 128, 8, True),
]
BLOCK = [  # B, H, Hkv, Sq, Sk, D, q_pos0, k_pos0, causal
    (1, 3, 3, 128, 384, 64, 256, 128, True),
    (2, 2, 1, 256, 256, 128, 0, 256, True),
]
BWD = [
    (1, 3, 1, 640, 64, 5, True),
    (2, 2, 2, 384, 128, 3, False),
]
MERGE = [  # n, B, S, H, D
    (3, 1, 5, 3, 8),
    (5, 1, 33, 2, 128),
    (2, 1, 3, 4500, 8),  # n*H past the tile budget: the row-per-thread kernel
]
SENTINEL = 7.0


def run_all(res):
    for i, (B, H, Hkv, S, D, P, causal) in enumerate(FWD):
        q, k, v = (t.cuda() for t in make_inputs(Workload("dbg", B, H, Hkv, S, D, P, causal), seed=3))
        out, lse = ra.ra_fwd(q, k, v, P=P, causal=causal)
        res[f"fwd{i}"] = (out.cpu(), lse.cpu(), ra.ra_get_last_device_status())
    for i, (B, H, Hkv, Sq, Sk, D, qp, kp, causal) in enumerate(BLOCK):
        g = torch.Generator().manual_seed(17 + i)
        q = torch.randn(B, Sq, H, D, generator=g).bfloat16().cuda()
        k = torch.randn(B, Sk, Hkv, D, generator=g).bfloat16().cuda()
        v = torch.randn(B, Sk, Hkv, D, generator=g).bfloat16().cuda()
        out, lse = ra.ra_fwd_block(q, k, v, q_pos0=qp, k_pos0=kp, causal=causal)
        res[f"block{i}"] = (out.cpu(), lse.cpu(), ra.ra_get_last_device_status())
    for i, (B, H, Hkv, S, D, P, causal) in enumerate(BWD):
        q, k, v = (t.cuda() for t in make_inputs(Workload("dbg", B, H, Hkv, S, D, P, causal), seed=5))
        out, lse = ra.ra_fwd(q, k, v, P=P, causal=causal)
        do = torch.randn(q.shape, generator=torch.Generator().manual_seed(9)).bfloat16().cuda()
        dq, dk, dv = ra.ra_bwd(q, k, v, out, lse, do, P=P, causal=causal)
        st = ra.ra_get_last_device_status()
        dq2, dk2, dv2 = (torch.empty_like(t) for t in (q, k, v))
        ra.ra_bwd_static(q, k, v, out, lse, do, dq2, dk2, dv2, P=P, causal=causal)
        res[f"bwd{i}"] = (dq.cpu(), dk.cpu(), dv.cpu(), st)
        res[f"bwd_static{i}"] = (dq2.cpu(), dk2.cpu(), dv2.cpu(), ra.ra_get_last_device_status())
    for i, (n, B, S, H, D) in enumerate(MERGE):
        for dt in (torch.bfloat16, torch.float32):
            g = torch.Generator().manual_seed(31 + i)
            o = torch.randn(n, B, S, H, D, generator=g).to(dt).cuda()
            l = (torch.randn(n, B, H, S, generator=g) * 3).cuda()
            l[0, 0, 0, 0] = -float("inf")
            out, lse = ra.ra_merge_partials(o, l)
            res[f"merge{i}_{str(dt)[6:]}"] = (out.cpu(), lse.cpu(), ra.ra_get_last_device_status())


def run_trim(res):
    """The test hook: the last `trim` elements of every buffer count as
    outside it, so the checks must fire and skip exactly those stores."""
    B, H, Hkv, S, D, P, causal = FWD[2]
    q, k, v = (t.cuda() for t in make_inputs(Workload("dbg", B, H, Hkv, S, D, P, causal), seed=3))
    trim = 3 * D
    out = torch.full((B, S, H, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, S), SENTINEL, dtype=torch.float32, device="cuda")
    ra.ra_debug_set_bounds_trim(trim)
    try:
        ra.ra_fwd(q, k, v, P=P, causal=causal, out=out, lse=lse)
        st_fwd = ra.ra_get_last_device_status()
        do = torch.randn(q.shape, generator=torch.Generator().manual_seed(9)).bfloat16().cuda()
        ra.ra_bwd(q, k, v, out, lse, do, P=P, causal=causal)
        st_bwd = ra.ra_get_last_device_status()
        n, Bm, Sm, Hm, Dm = MERGE[1]
        g = torch.Generator().manual_seed(32)
        o = torch.randn(n, Bm, Sm, Hm, Dm, generator=g).bfloat16().cuda()
        lp = (torch.randn(n, Bm, Hm, Sm, generator=g) * 3).cuda()
        mout = torch.full((Bm, Sm, Hm, Dm), SENTINEL, dtype=torch.bfloat16, device="cuda")
        mlse = torch.full((Bm, Hm, Sm), SENTINEL, dtype=torch.float32, device="cuda")
        ra.ra_merge_partials(o, lp, out=mout, lse=mlse)
        st_merge = ra.ra_get_last_device_status()
    finally:
        ra.ra_debug_set_bounds_trim(0)
    out0, lse0 = ra.ra_fwd(q, k, v, P=P, causal=causal)
    res["trim"] = dict(trim=trim, st_fwd=st_fwd, st_bwd=st_bwd, st_merge=st_merge,
                       out=out.cpu(), lse=lse.cpu(), out0=out0.cpu(), lse0=lse0.cpu(),
                       mout=mout.cpu(), mlse=mlse.cpu(), sentinel=SENTINEL)


if __name__ == "__main__":
    res = {"debug_build": ra.ra_debug_build()}
    run_all(res)
    if "--trim" in sys.argv:
        run_trim(res)
    torch.save(res, sys.argv[1])
