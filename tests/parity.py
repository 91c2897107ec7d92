"""Comparison helpers for GPU-vs-oracle parity (tolerances of the method's
accuracy target: bf16 O within 1.5e-2 max-abs and 2e-3 mean-abs of the fp64
oracle for V ~ N(0,1); LSE within 1e-3 relative, read as
|d lse| <= 1e-3 * max(1, |lse|) so that rows with lse near 0 stay meaningful)."""
import numpy as np
import torch

MAX_ABS = 1.5e-2
MEAN_ABS = 2e-3
LSE_REL = 1e-3


def rows_to_bhs(rows, H, S):
    rows = np.asarray(rows, dtype=np.int64)
    s = rows % S
    h = (rows // S) % H
    b = rows // (S * H)
    return b, h, s


def compare(out_gpu, lse_gpu, out_ref, lse_ref, rows=None):
    """out_gpu [B,S,H,D] bf16 (torch, any device), lse_gpu [B,H,S] fp32.
    out_ref/lse_ref: full arrays ([B,S,H,D], [B,H,S]) or sampled rows
    ([n,D], [n]) with ``rows`` flat ids.  Returns a stats dict."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64) if lse_gpu is not None else None
    if rows is not None:
        B, S, H, D = o.shape
        b, h, s = rows_to_bhs(rows, H, S)
        o = o[b, s, h]
        if l is not None:
            l = l[b, h, s]
    err = np.abs(o - out_ref)
    st = {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
          "finite": bool(np.isfinite(o).all())}
    # error of the ideal bf16 rounding of the oracle, for attribution
    ref_bf16 = torch.tensor(out_ref).to(torch.bfloat16).double().numpy()
    st["max_abs_vs_rounded_ref"] = float(np.abs(o - ref_bf16).max())
    st["n_ref_ge4_at_max"] = int(((err > MAX_ABS) & (np.abs(out_ref) >= 4)).sum())
    if l is not None:
        dl = np.abs(l - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
        st["lse_rel"] = float(dl.max())
    return st


def assert_parity(st, what=""):
    assert st["finite"], f"{what}: non-finite output"
    assert st["max_abs"] <= MAX_ABS, f"{what}: max-abs {st['max_abs']:.3e} > {MAX_ABS} ({st})"
    assert st["mean_abs"] <= MEAN_ABS, f"{what}: mean-abs {st['mean_abs']:.3e} > {MEAN_ABS} ({st})"
    if "lse_rel" in st:
        assert st["lse_rel"] <= LSE_REL, f"{what}: lse rel {st['lse_rel']:.3e} > {LSE_REL} ({st})"
