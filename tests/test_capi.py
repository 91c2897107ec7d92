"""C-ABI checks that need no GPU: the library loads, exports every function
``include/ringattn.h`` declares, and host-side validation rejects bad
arguments before touching the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ringattn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("ra_fwd", "ra_merge_partials", "ra_bwd", "ra_bwd_workspace_bytes",
              "ra_get_last_device_status", "ra_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(ralib):
    lib = ctypes.CDLL(ralib.library_path())
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings(ralib):
    assert ralib.ra_status_string(0) == "RA_OK"
    assert ralib.ra_status_string(4) == "RA_ERR_TIMEOUT"
    assert ralib.ra_status_string(99) == "RA_ERR_UNKNOWN"
    assert ralib.ra_version() == (0 << 16) | (3 << 8)


# Fake, 16-byte aligned addresses: validation must reject these calls before
# any CUDA call, so the addresses are never dereferenced.
Q, K, V, O, L = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
OK_SHAPE = dict(B=1, H=4, Hkv=2, S=256, D=128, P=2, causal=1, scale=0.125)


def _call(ralib, q=Q, k=K, v=V, o=O, l=L, **kw):
    a = dict(OK_SHAPE)
    a.update(kw)
    return ralib.ra_fwd_raw(q, k, v, o, l, a["B"], a["H"], a["Hkv"], a["S"], a["D"], a["P"],
                            a["causal"], a["scale"], stream=0)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(o=0), 1),
    (dict(B=0), 1), (dict(H=-1), 1), (dict(S=0), 1), (dict(D=0), 1), (dict(P=0), 1),
    (dict(H=3, Hkv=2), 1),             # H % Hkv != 0
    (dict(S=256, P=3), 1),             # S % P != 0
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(scale=-0.5), 2),             # negative scale: outside the kernels
    (dict(D=96), 2), (dict(D=256), 2),
    (dict(S=384, P=2), 2),             # chunk of 192 rows: not a multiple of 128
    (dict(S=200, P=1), 2),             # ragged sequence
    (dict(q=Q + 8), 2), (dict(o=O + 4), 2), (dict(l=L + 2), 2),
    (dict(B=1 << 16, S=1 << 15, P=1), 2),  # B*S >= 2^31 rows
    (dict(H=1 << 13, S=1 << 24, P=1), 2),  # 2^30 query tiles: work-item ids must stay in int
])
def test_fwd_validation_rejects_before_launch(ralib, kw, code):
    assert _call(ralib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(o=0), 1), (dict(l=0), 1), (dict(out=0), 1), (dict(n=0), 1), (dict(B=0), 1),
    (dict(D=12), 2), (dict(o=O + 8), 2), (dict(out=O + 8), 2),
])
def test_merge_validation_rejects_before_launch(ralib, kw, code):
    a = dict(o=Q, l=L, n=2, out=O, lse=L + 4096, B=1, H=2, S=128, D=64)
    a.update(kw)
    lib = ralib._load()
    rc = lib.ra_merge_partials(a["o"], 0, a["l"], a["n"], a["out"], a["lse"], a["B"], a["H"],
                               a["S"], a["D"], None)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(Sk=0), 1), (dict(qp=-128), 1), (dict(kp=-128), 1),
    (dict(H=3, Hkv=2), 1), (dict(scale=float("nan")), 1),
    (dict(Sq=200), 2), (dict(Sk=100), 2), (dict(qp=64), 2), (dict(kp=1), 2), (dict(D=32), 2),
    (dict(scale=-1.0), 2), (dict(o=O + 4), 2),
    (dict(H=1 << 13, Sq=1 << 24), 2),  # 2^30 query tiles
])
def test_block_validation_rejects_before_launch(ralib, kw, code):
    a = dict(q=Q, k=K, v=V, o=O, l=L, B=1, H=4, Hkv=2, Sq=256, Sk=384, D=128, qp=256, kp=0,
             causal=1, scale=0.125)
    a.update(kw)
    lib = ralib._load()
    rc = lib.ra_fwd_block(a["q"], a["k"], a["v"], a["o"], a["l"], a["B"], a["H"], a["Hkv"], a["Sq"],
                          a["Sk"], a["D"], a["qp"], a["kp"], a["causal"], a["scale"], None)
    assert rc == code


def test_bwd_workspace_bytes(ralib):
    assert ralib.ra_bwd_workspace_bytes(2, 32, 16384) == 8 * 2 * 32 * 16384
    assert ralib.ra_bwd_workspace_bytes(0, 4, 128) == 0
    assert ralib.ra_bwd_workspace_bytes(1, -1, 128) == 0


W = 0x60000
@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(lse=0), 1), (dict(dout=0), 1), (dict(dq=0), 1), (dict(dk=0), 1),
    (dict(dv=0), 1), (dict(ws=0), 1), (dict(B=0), 1), (dict(P=3), 1), (dict(H=3, Hkv=2), 1),
    (dict(scale=float("nan")), 1),
    (dict(ws_bytes=8 * 4 * 256 - 16), 1),    # one row short of 8*B*H*S
    (dict(scale=-0.1), 2), (dict(D=96), 2), (dict(S=384, P=2, ws_bytes=8 * 4 * 384), 2),
    (dict(dq=O + 8), 2), (dict(ws=W + 4), 2), (dict(lse=L + 2), 2),
])
def test_bwd_validation_rejects_before_launch(ralib, kw, code):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, dout=Q + 0x100000, dq=O + 0x100000, dk=K + 0x100000,
             dv=V + 0x100000, ws=W, ws_bytes=8 * 4 * 256, B=1, H=4, Hkv=2, S=256, D=128, P=2,
             causal=1, scale=0.125)
    a.update(kw)
    lib = ralib._load()
    rc = lib.ra_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dout"], a["dq"], a["dk"], a["dv"],
                    a["ws"], a["ws_bytes"], a["B"], a["H"], a["Hkv"], a["S"], a["D"], a["P"],
                    a["causal"], a["scale"], None)
    assert rc == code


def test_binding_rejects_tensors_it_cannot_hand_to_the_device(ralib):
    """The binding passes raw addresses, so a tensor that is not a CUDA tensor
    on the inputs' device, or has the wrong rank, must be refused before any
    CUDA call (on a host without a GPU every tensor here is a CPU tensor)."""
    import torch

    q = torch.zeros(1, 256, 2, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 256)
    with pytest.raises(ValueError):
        ralib.ra_fwd(q, q, q, P=1, causal=True)
    with pytest.raises(ValueError):
        ralib.ra_fwd(q[0], q, q, P=1, causal=True)  # 3-D q
    with pytest.raises(ValueError):
        ralib.ra_fwd_block(q, q, q, q_pos0=0, k_pos0=0, causal=True)
    with pytest.raises(ValueError):
        ralib.ra_bwd(q, q, q, q, lse, q, P=1, causal=True)
    with pytest.raises(ValueError):
        ralib.ra_bwd_static(q, q, q, q, lse, q, q, q, q, P=1, causal=True)
    with pytest.raises(ValueError):
        ralib.ra_merge_partials(q[None], lse[None])
    with pytest.raises(ValueError):
        ralib.ra_merge_partials(q, lse)  # 4-D partials
