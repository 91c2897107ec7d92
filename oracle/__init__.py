"""fp64 CPU oracle for ring-chunked attention (forward, and its gradients).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and ``bench.py``'s CPU-baseline / reference arm may import
this package.  It shares no code with the CUDA path; the two meet only in the
seeded input generator (``ring_chunked_attention_gb300.inputs``), which holds
none of the method's arithmetic.

Source of the definition: the mKernel overview page (chatgpz.de, German
translation of the MarkTechPost article), table "Die fünf verschmolzenen
Kerne", row "Ring Attention": the local computation is FlashAttention (exact
softmax attention) and the key/value blocks arrive in ring order and are folded
one at a time.  ``ora.c`` carries the formulas.

Every function pins down its part of the method against something other than
itself in ``tests/test_oracle_pins.py`` (closed forms, hand-derived fixtures
under ``tests/golden/``, invariants, brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ora.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ora.c`` with gcc into ``liboracle.so`` (plain -O2, no
    fast-math, no contraction, portable across x86_64 and aarch64)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # RA_ORACLE_LIB lets the mutation test load a deliberately broken
        # build of ora.c to show that the pins catch it.
        path = os.environ.get("RA_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64p = ctypes.POINTER(ctypes.c_int64)
        f64p = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.ora_attn_direct.argtypes = [u16p, u16p, u16p, i, i, i, i, i, i,
                                        ctypes.c_double, i64p, ctypes.c_int64,
                                        f64p, f64p, f64p, i]
        lib.ora_attn_direct.restype = i
        lib.ora_attn_ring.argtypes = [u16p, u16p, u16p, i, i, i, i, i, i, i,
                                      ctypes.c_double, i64p, ctypes.c_int64,
                                      f64p, f64p, i]
        lib.ora_attn_ring.restype = i
        lib.ora_attn_block.argtypes = [u16p, u16p, u16p, i, i, i, i, i, i, ctypes.c_longlong,
                                       ctypes.c_longlong, i, ctypes.c_double, f64p, f64p]
        lib.ora_attn_block.restype = i
        lib.ora_merge.argtypes = [f64p, f64p, i, i, i, i, i, f64p, f64p]
        lib.ora_merge.restype = i
        lib.ora_attn_bwd.argtypes = [u16p, u16p, u16p, u16p, u16p, i, i, i, i, i, i,
                                     ctypes.c_double, f64p, f64p, f64p, i]
        lib.ora_attn_bwd.restype = i
        lib.ora_attn_bwd_dq.argtypes = [u16p, u16p, u16p, u16p, u16p, i, i, i, i, i, i,
                                        ctypes.c_double, i64p, ctypes.c_int64, f64p, i]
        lib.ora_attn_bwd_dq.restype = i
        lib.ora_default_threads.argtypes = []
        lib.ora_default_threads.restype = i
        _lib = lib
    return _lib


def default_threads() -> int:
    """Threads the oracle uses when asked for 0: every online host core."""
    return int(_load().ora_default_threads())


def _bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 bit patterns."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16, "numpy inputs must be bf16 bit patterns (uint16)"
        return np.ascontiguousarray(x)
    import torch  # CPU only: used to reinterpret bf16 storage

    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _shapes(q, k, v):
    B, S, H, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    assert (Bk, Sk, Dk) == (B, S, D) and tuple(v.shape) == tuple(k.shape)
    return B, S, H, Hkv, D


def attn_direct(q, k, v, causal: bool, scale: float, rows=None, threads: int = 0,
                return_weights: bool = False):
    """Two-pass definition.  ``rows``: optional int64 flat ids
    ``(b*H + h)*S + s``.  Returns ``out`` [n_rows, D] and ``lse`` [n_rows]
    (all rows: reshaped to [B,S,H,D] and [B,H,S]), plus the weights
    [n_rows, S] if asked."""
    B, S, H, Hkv, D = _shapes(q, k, v)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    n = B * H * S if rows is None else len(rows)
    out = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    w = np.empty((n, S), np.float64) if return_weights else None
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    rc = _load().ora_attn_direct(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        B, H, Hkv, S, D, int(bool(causal)), float(scale),
        None if rows_a is None else _ptr(rows_a, ctypes.c_int64), n,
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
        None if w is None else _ptr(w, ctypes.c_double), int(threads))
    if rc != 0:
        raise ValueError(f"ora_attn_direct failed ({rc})")
    if rows is None:
        out = out.reshape(B, H, S, D).transpose(0, 2, 1, 3).copy()
        lse = lse.reshape(B, H, S)
    return (out, lse, w) if return_weights else (out, lse)


def attn_ring(q, k, v, P: int, causal: bool, scale: float, rows=None, threads: int = 0):
    """Chunk-by-chunk fold in ring order (see ``ora.c``).  Same return
    convention as :func:`attn_direct`."""
    B, S, H, Hkv, D = _shapes(q, k, v)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    n = B * H * S if rows is None else len(rows)
    out = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    rc = _load().ora_attn_ring(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        B, H, Hkv, S, D, int(P), int(bool(causal)), float(scale),
        None if rows_a is None else _ptr(rows_a, ctypes.c_int64), n,
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), int(threads))
    if rc != 0:
        raise ValueError(f"ora_attn_ring failed ({rc})")
    if rows is None:
        out = out.reshape(B, H, S, D).transpose(0, 2, 1, 3).copy()
        lse = lse.reshape(B, H, S)
    return out, lse


def attn_block(q, k, v, q_pos0: int, k_pos0: int, causal: bool, scale: float):
    """One ring step: q [B,Sq,H,D] (global rows q_pos0..) against k/v
    [B,Sk,Hkv,D] (global rows k_pos0..).  Returns out [B,Sq,H,D] and lse
    [B,H,Sq]; rows with no allowed key give 0 and -inf."""
    B, Sq, H, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    assert Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    out = np.empty((B, Sq, H, D), np.float64)
    lse = np.empty((B, H, Sq), np.float64)
    rc = _load().ora_attn_block(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                _ptr(vb, ctypes.c_uint16), B, H, Hkv, Sq, Sk, D, int(q_pos0),
                                int(k_pos0), int(bool(causal)), float(scale),
                                _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"ora_attn_block failed ({rc})")
    return out, lse


def merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge normalised partials: ``o_parts`` [n,B,S,H,D], ``lse_parts``
    [n,B,H,S] (any float dtype, widened exactly to fp64)."""
    o = np.ascontiguousarray(o_parts, dtype=np.float64)
    l = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, B, S, H, D = o.shape
    assert l.shape == (n, B, H, S)
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    rc = _load().ora_merge(_ptr(o, ctypes.c_double), _ptr(l, ctypes.c_double), n, B, H, S, D,
                           _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"ora_merge failed ({rc})")
    return out, lse


def attn_bwd(q, k, v, dout, causal: bool, scale: float, out=None, threads: int = 0):
    """Gradients of ``sum(out * dout)`` for the attention above (the
    derivative of the definition; see ``ora.c``).  ``out``: optional bf16
    forward output [B,S,H,D] that delta = <dout, out> is taken from (exact
    delta when None).  Returns fp64 ``dq`` [B,S,H,D], ``dk`` and ``dv``
    [B,S,Hkv,D]."""
    B, S, H, Hkv, D = _shapes(q, k, v)
    assert tuple(dout.shape) == tuple(q.shape)
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    ob = None if out is None else _bits(out)
    assert ob is None or ob.shape == tuple(q.shape)
    dq = np.empty((B, S, H, D), np.float64)
    dk = np.empty((B, S, Hkv, D), np.float64)
    dv = np.empty((B, S, Hkv, D), np.float64)
    rc = _load().ora_attn_bwd(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        _ptr(db, ctypes.c_uint16), None if ob is None else _ptr(ob, ctypes.c_uint16), B, H, Hkv, S, D, int(bool(causal)), float(scale),
        _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
        int(threads))
    if rc != 0:
        raise ValueError(f"ora_attn_bwd failed ({rc})")
    return dq, dk, dv


def attn_bwd_dq(q, k, v, dout, causal: bool, scale: float, rows, out_rows=None,
                threads: int = 0):
    """``dq`` of selected query rows (flat ids ``(b*H + h)*S + s``), [n, D].
    ``out_rows``: optional bf16 forward output of those rows [n, D] that
    delta is taken from (exact delta when None)."""
    B, S, H, Hkv, D = _shapes(q, k, v)
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    rows_a = np.ascontiguousarray(rows, dtype=np.int64)
    ob = None if out_rows is None else _bits(out_rows)
    assert ob is None or ob.shape == (len(rows_a), D)
    dq = np.empty((len(rows_a), D), np.float64)
    rc = _load().ora_attn_bwd_dq(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        _ptr(db, ctypes.c_uint16), None if ob is None else _ptr(ob, ctypes.c_uint16), B, H, Hkv, S,
        D, int(bool(causal)), float(scale), _ptr(rows_a, ctypes.c_int64), len(rows_a), _ptr(dq, ctypes.c_double), int(threads))
    if rc != 0:
        raise ValueError(f"ora_attn_bwd_dq failed ({rc})")
    return dq


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
