"""Guard bands around every output buffer, for every entry point.

compute-sanitizer is not available, so out-of-bounds writes are caught the
plain way: each output (and the backward's workspace) is carved out of a
larger device buffer whose bytes before and after it hold a poison pattern,
the call runs, and the pattern must be intact afterwards.  Inputs are
compared with copies taken before the call (the kernels only read them).
The shapes are the awkward ones: one 128-row tile per chunk (P = S/128),
fewer (b, h) pairs than SMs, odd head counts, block offsets, a merge with a
row length that is not a multiple of the 16-byte vector width of a row group.
"""
import pytest
import torch

from ring_chunked_attention_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes of poison on each side (a multiple of 16: alignment kept)
POISON = 0xA5


class Guarded:
    """Device tensors of the given shapes/dtypes, each inside its own buffer
    with GUARD poisoned bytes before and after it."""

    def __init__(self):
        self.bufs = []

    def alloc(self, shape, dtype):
        n = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((GUARD + n + GUARD,), POISON, dtype=torch.uint8, device="cuda")
        t = buf[GUARD:GUARD + n].view(dtype).view(shape)
        t.fill_(0)
        self.bufs.append(buf)
        return t

    def intact(self):
        torch.cuda.synchronize()
        for buf in self.bufs:
            head, tail = buf[:GUARD], buf[-GUARD:]
            if not (bool((head == POISON).all()) and bool((tail == POISON).all())):
                return False
        return True


def _inputs(w, seed):
    return tuple(t.cuda() for t in make_inputs(w, seed=seed))


FWD_SHAPES = [
    # B, H, Hkv, S, D, P, causal
    (1, 3, 1, 640, 64, 5, True),      # one tile per chunk, 3 query heads
    (2, 5, 5, 384, 128, 3, False),    # odd heads, non-causal, B*H < SMs
    (1, 4, 2, 1024, 128, 8, True),    # GQA pairs of heads
    (3, 1, 1, 256, 64, 2, True),      # single head, several batch entries
]


@pytest.mark.parametrize("shape", FWD_SHAPES, ids=[str(s) for s in FWD_SHAPES])
@pytest.mark.parametrize("pairing", [0, 1, 2], ids=["auto", "paired", "single"])
def test_fwd_writes_nothing_outside_out_and_lse(ralib, cuda_ok, shape, pairing):
    B, H, Hkv, S, D, P, causal = shape
    w = Workload("canary", B, H, Hkv, S, D, P, causal)
    q, k, v = _inputs(w, 3)
    keep = [t.clone() for t in (q, k, v)]
    gd = Guarded()
    out = gd.alloc((B, S, H, D), torch.bfloat16)
    lse = gd.alloc((B, H, S), torch.float32)
    ralib.ra_set_item_pairing(pairing)
    try:
        ralib.ra_fwd(q, k, v, P=P, causal=causal, out=out, lse=lse)
    finally:
        ralib.ra_set_item_pairing(0)
    assert gd.intact()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    assert all(torch.equal(a, b) for a, b in zip((q, k, v), keep))
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()


BLOCK_CASES = [
    # B, H, Hkv, Sq, Sk, D, q_pos0, k_pos0, causal
    (1, 3, 3, 128, 384, 64, 256, 128, True),   # straddles the diagonal
    (2, 2, 1, 256, 256, 128, 0, 256, True),    # every row empty (all keys in the future)
    (1, 5, 5, 384, 128, 128, 640, 0, False),
]


@pytest.mark.parametrize("case", BLOCK_CASES, ids=[str(c) for c in BLOCK_CASES])
def test_fwd_block_writes_nothing_outside_out_and_lse(ralib, cuda_ok, case):
    B, H, Hkv, Sq, Sk, D, qp, kp, causal = case
    g = torch.Generator().manual_seed(sum(case[:6]))
    q = torch.randn(B, Sq, H, D, generator=g).bfloat16().cuda()
    k = torch.randn(B, Sk, Hkv, D, generator=g).bfloat16().cuda()
    v = torch.randn(B, Sk, Hkv, D, generator=g).bfloat16().cuda()
    gd = Guarded()
    out = gd.alloc((B, Sq, H, D), torch.bfloat16)
    lse = gd.alloc((B, H, Sq), torch.float32)
    ralib.ra_fwd_block(q, k, v, q_pos0=qp, k_pos0=kp, causal=causal, out=out, lse=lse)
    assert gd.intact()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK


BWD_SHAPES = [
    (1, 3, 1, 640, 64, 5, True),
    (2, 2, 2, 384, 128, 3, False),
    (1, 4, 2, 512, 128, 4, True),
]


@pytest.mark.parametrize("shape", BWD_SHAPES, ids=[str(s) for s in BWD_SHAPES])
@pytest.mark.parametrize("entry", ["ra_bwd", "ra_bwd_static"])
def test_bwd_writes_nothing_outside_its_outputs(ralib, cuda_ok, shape, entry):
    B, H, Hkv, S, D, P, causal = shape
    w = Workload("canary", B, H, Hkv, S, D, P, causal)
    q, k, v = _inputs(w, 5)
    out, lse = ralib.ra_fwd(q, k, v, P=P, causal=causal)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(9)).bfloat16().cuda()
    keep = [t.clone() for t in (q, k, v, out, lse, do)]
    gd = Guarded()
    dq = gd.alloc(q.shape, torch.bfloat16)
    dk = gd.alloc(k.shape, torch.bfloat16)
    dv = gd.alloc(v.shape, torch.bfloat16)
    if entry == "ra_bwd":
        ws = gd.alloc((ralib.ra_bwd_workspace_bytes(B, H, S),), torch.uint8)
        ralib.ra_bwd(q, k, v, out, lse, do, P=P, causal=causal, dq=dq, dk=dk, dv=dv, workspace=ws)
    else:
        ralib.ra_bwd_static(q, k, v, out, lse, do, dq, dk, dv, P=P, causal=causal)
    assert gd.intact()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    assert all(torch.equal(a, b) for a, b in zip((q, k, v, out, lse, do), keep))
    assert all(torch.isfinite(t).all() for t in (dq, dk, dv))


MERGE_SHAPES = [
    # n, B, S, H, D
    (3, 1, 5, 3, 8),       # one 16-byte group per row, ragged row count
    (2, 2, 7, 1, 24),      # D not a power of two
    (5, 1, 33, 2, 128),
]


@pytest.mark.parametrize("shape", MERGE_SHAPES, ids=[str(s) for s in MERGE_SHAPES])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_merge_writes_nothing_outside_out_and_lse(ralib, cuda_ok, shape, dtype):
    n, B, S, H, D = shape
    g = torch.Generator().manual_seed(sum(shape))
    o = torch.randn(n, B, S, H, D, generator=g).to(dtype).cuda()
    l = (torch.randn(n, B, H, S, generator=g) * 3).cuda()
    l[0, 0, 0, 0] = -float("inf")
    keep = [o.clone(), l.clone()]
    gd = Guarded()
    out = gd.alloc((B, S, H, D), torch.bfloat16)
    lse = gd.alloc((B, H, S), torch.float32)
    ralib.ra_merge_partials(o, l, out=out, lse=lse)
    assert gd.intact()
    assert torch.equal(o, keep[0]) and torch.equal(l, keep[1])
