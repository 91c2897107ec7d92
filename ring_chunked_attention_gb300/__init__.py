"""ring_chunked_attention_gb300 -- Python binding of libringattn.

The compute path is the C ABI in ``include/ringattn.h`` (CUDA kernels for
sm_103a).  This module only marshals arguments: it takes torch tensors for
device memory and streams, checks shapes/dtypes, and passes raw pointers to
the library.  There is no fallback: if ``libringattn.so`` is missing or
cannot be loaded, every call raises.

Functions carry the C names:

* :func:`ra_fwd` -- ring-chunked attention forward (out, lse);
* :func:`ra_fwd_block` -- one ring step (a query block against a key/value block);
* :func:`ra_bwd` -- gradients dq, dk, dv of the forward for a given dout;
* :func:`ra_merge_partials` -- merge normalised partials over disjoint key sets;
* :func:`ra_get_last_device_status`, :func:`ra_status_string`,
  :func:`ra_debug_set_fault`, :func:`ra_shutdown`.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["ra_fwd", "ra_fwd_block", "ra_bwd", "ra_bwd_static", "ra_bwd_workspace_bytes", "ra_merge_partials", "ra_measure_ceilings", "ra_get_last_device_status", "ra_status_string",
           "ra_debug_set_fault", "ra_set_mma_order", "ra_set_item_pairing", "ra_shutdown", "ra_version",
           "RaError", "library_path", "MMA_ORDER_GROUPED", "MMA_ORDER_STRICT", "MMA_ORDER_INORDER",
           "MMA_ORDER_BRIDGED",
           "RA_OK", "RA_ERR_INVALID_ARG", "RA_ERR_UNSUPPORTED", "RA_ERR_CUDA", "RA_ERR_TIMEOUT",
           "RA_ERR_BOUNDS", "ra_debug_build", "ra_debug_set_bounds_trim", "ra_trace_build",
           "ra_trace_read"]

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_TIMEOUT, RA_ERR_BOUNDS = (
    0, 1, 2, 3, 4, 5)

_HERE = os.path.dirname(os.path.abspath(__file__))
# RA_DEBUG=1 selects the bounds-checked build (python -m ring_chunked_attention_gb300.build --debug),
# RA_TRACE=1 the traced one (--trace)
_DEBUG = os.environ.get("RA_DEBUG", "0") == "1"
_TRACE = os.environ.get("RA_TRACE", "0") == "1" and not _DEBUG
_LIB_PATH = os.path.join(_HERE, "libringattn_debug.so" if _DEBUG else
                         "libringattn_trace.so" if _TRACE else "libringattn.so")
_lib = None

EXPORTS = ("ra_fwd", "ra_fwd_block", "ra_bwd", "ra_bwd_static", "ra_bwd_workspace_bytes", "ra_merge_partials", "ra_measure_ceilings", "ra_get_last_device_status", "ra_status_string",
           "ra_last_cuda_error", "ra_version", "ra_debug_set_fault", "ra_set_mma_order",
           "ra_set_item_pairing", "ra_shutdown", "ra_debug_build", "ra_debug_set_bounds_trim",
           "ra_trace_read")


class RaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {ra_status_string(code)}"
                         + (f" (cudaError {_load().ra_last_cuda_error()})" if code == RA_ERR_CUDA else ""))


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{os.path.basename(_LIB_PATH)} is not built ({_LIB_PATH}); run "
                           "`python -m ring_chunked_attention_gb300.build`"
                           + (" --debug" if _DEBUG else " --trace" if _TRACE else ""))
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.ra_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.ra_fwd.restype = i
    ll = ctypes.c_longlong
    lib.ra_fwd_block.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ll, ll, i, f, vp]
    lib.ra_fwd_block.restype = i
    ull = ctypes.c_ulonglong
    lib.ra_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.ra_bwd_workspace_bytes.restype = ull
    lib.ra_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ull, i, i, i, i, i, i, i, f, vp]
    lib.ra_bwd.restype = i
    lib.ra_bwd_static.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.ra_bwd_static.restype = i
    lib.ra_merge_partials.argtypes = [vp, i, vp, i, vp, vp, i, i, i, i, vp]
    lib.ra_merge_partials.restype = i
    lib.ra_measure_ceilings.argtypes = [ctypes.POINTER(ctypes.c_double)]
    lib.ra_measure_ceilings.restype = i
    lib.ra_get_last_device_status.argtypes = [vp]
    lib.ra_get_last_device_status.restype = i
    lib.ra_status_string.argtypes = [i]
    lib.ra_status_string.restype = ctypes.c_char_p
    lib.ra_last_cuda_error.argtypes = []
    lib.ra_last_cuda_error.restype = i
    lib.ra_version.argtypes = []
    lib.ra_version.restype = i
    lib.ra_debug_set_fault.argtypes = [ctypes.c_longlong, i]
    lib.ra_debug_set_fault.restype = None
    lib.ra_set_mma_order.argtypes = [i]
    lib.ra_set_mma_order.restype = None
    lib.ra_set_item_pairing.argtypes = [i]
    lib.ra_set_item_pairing.restype = None
    lib.ra_shutdown.argtypes = []
    lib.ra_shutdown.restype = None
    lib.ra_debug_build.argtypes = []
    lib.ra_debug_build.restype = i
    lib.ra_debug_set_bounds_trim.argtypes = [ctypes.c_longlong]
    lib.ra_debug_set_bounds_trim.restype = None
    lib.ra_trace_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i]
    lib.ra_trace_read.restype = i
    _lib = lib
    return lib


def _stream_ptr(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _check(code: int, what: str):
    if code != RA_OK:
        raise RaError(code, what)


def _dims(t, name: str, ndim: int):
    """Shape of a tensor argument that must have ``ndim`` dimensions."""
    import torch

    if not isinstance(t, torch.Tensor) or t.dim() != ndim:
        raise ValueError(f"{name} must be a {ndim}-D tensor")
    return tuple(t.shape)


def _tensor_checks(device, *specs):
    """Each spec is (tensor, name, dtypes, shape or None).  The library reads
    and writes these tensors by address on one device, so each must be a
    contiguous CUDA tensor on ``device`` with one of the dtypes and the shape."""
    import torch

    for t, name, dtypes, shape in specs:
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != device:
            raise ValueError(f"{name} must be a CUDA tensor on {device}")
        if t.dtype not in dtypes:
            raise ValueError(f"{name} must have dtype {' or '.join(str(d) for d in dtypes)}, "
                             f"got {t.dtype}")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def _call_on(device, stream, fn):
    """Run ``fn(stream_handle)`` with ``device`` current: the library launches
    on the current device.  ``stream`` (default: that device's current
    stream) must belong to the same device."""
    import torch

    with torch.cuda.device(device):
        if stream is not None and hasattr(stream, "device") and stream.device != device:
            raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
        return fn(_stream_ptr(stream))


def ra_status_string(code: int) -> str:
    return _load().ra_status_string(int(code)).decode()


def ra_version() -> int:
    return int(_load().ra_version())


def ra_fwd(q, k, v, *, P: int, causal: bool, scale: float | None = None, out=None, lse=None,
           want_lse: bool = True, stream=None):
    """Ring-chunked attention forward.  ``q`` [B,S,H,D], ``k``/``v``
    [B,S,Hkv,D] bf16 CUDA tensors (contiguous, one device).  Returns
    ``(out, lse)`` with ``out`` [B,S,H,D] bf16 and ``lse`` [B,H,S] fp32
    (``None`` when ``want_lse`` is false and no ``lse`` buffer is given).
    ``scale`` defaults to 1/sqrt(D)."""
    import torch

    lib = _load()
    B, S, H, D = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[2]
    dev, bf = q.device, (torch.bfloat16,)
    _tensor_checks(dev, (q, "q", bf, None), (k, "k", bf, (B, S, Hkv, D)),
                   (v, "v", bf, (B, S, Hkv, D)))
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    _tensor_checks(dev, (out, "out", bf, (B, S, H, D)))
    if lse is not None:
        _tensor_checks(dev, (lse, "lse", (torch.float32,), (B, H, S)))
    code = _call_on(dev, stream, lambda sp: lib.ra_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
        None if lse is None else lse.data_ptr(), B, H, Hkv, S, D, int(P), int(bool(causal)),
        float(scale), sp))
    _check(code, "ra_fwd")
    return out, lse


def ra_fwd_block(q, k, v, *, q_pos0: int, k_pos0: int, causal: bool, scale: float | None = None,
                 out=None, lse=None, want_lse: bool = True, stream=None):
    """One ring step: ``q`` [B,Sq,H,D] (global rows q_pos0..) against ``k``/``v``
    [B,Sk,Hkv,D] (global rows k_pos0..).  Returns the normalised partial
    ``(out [B,Sq,H,D] bf16, lse [B,H,Sq] fp32)``; rows with no allowed key get
    0 and -inf."""
    import torch

    lib = _load()
    B, Sq, H, D = _dims(q, "q", 4)
    _, Sk, Hkv, _ = _dims(k, "k", 4)
    dev, bf = q.device, (torch.bfloat16,)
    _tensor_checks(dev, (q, "q", bf, None), (k, "k", bf, (B, Sk, Hkv, D)),
                   (v, "v", bf, (B, Sk, Hkv, D)))
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    _tensor_checks(dev, (out, "out", bf, (B, Sq, H, D)))
    if lse is not None:
        _tensor_checks(dev, (lse, "lse", (torch.float32,), (B, H, Sq)))
    code = _call_on(dev, stream, lambda sp: lib.ra_fwd_block(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
        None if lse is None else lse.data_ptr(), B, H, Hkv, Sq, Sk, D, int(q_pos0), int(k_pos0),
        int(bool(causal)), float(scale), sp))
    _check(code, "ra_fwd_block")
    return out, lse


def ra_bwd_workspace_bytes(B: int, H: int, S: int) -> int:
    """Device workspace bytes :func:`ra_bwd` needs (8 * B * H * S)."""
    return int(_load().ra_bwd_workspace_bytes(int(B), int(H), int(S)))


def ra_bwd(q, k, v, out, lse, dout, *, P: int, causal: bool, scale: float | None = None,
           dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients of :func:`ra_fwd` for output gradient ``dout`` [B,S,H,D] bf16.
    ``out`` and ``lse`` are the forward's results for the same inputs and
    options.  Returns ``(dq, dk, dv)`` (bf16, shapes of q, k, v); buffers and
    the workspace are allocated with torch when not given."""
    import torch

    lib = _load()
    B, S, H, D = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[2]
    dev, bf = q.device, (torch.bfloat16,)
    _tensor_checks(dev, (q, "q", bf, None), (k, "k", bf, (B, S, Hkv, D)),
                   (v, "v", bf, (B, S, Hkv, D)), (out, "out", bf, (B, S, H, D)),
                   (dout, "dout", bf, (B, S, H, D)), (lse, "lse", (torch.float32,), (B, H, S)))
    if scale is None:
        scale = D ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _tensor_checks(dev, (dq, "dq", bf, (B, S, H, D)), (dk, "dk", bf, (B, S, Hkv, D)),
                   (dv, "dv", bf, (B, S, Hkv, D)))
    need = ra_bwd_workspace_bytes(B, H, S)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _tensor_checks(dev, (workspace, "workspace", (workspace.dtype,), None))
    code = _call_on(dev, stream, lambda sp: lib.ra_bwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
        dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), B, H, Hkv, S, D, int(P),
        int(bool(causal)), float(scale), sp))
    _check(code, "ra_bwd")
    return dq, dk, dv


def ra_bwd_static(q, k, v, out, lse, dout, dq, dk, dv, *, P: int, causal: bool,
                  scale: float | None = None, stream=None):
    """:func:`ra_bwd` on the library's fixed scratch (no workspace, no
    allocation in the call; calls that can overlap race on that scratch).
    The caller passes the output buffers ``dq``, ``dk``, ``dv``."""
    import torch

    lib = _load()
    B, S, H, D = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[2]
    dev, bf = q.device, (torch.bfloat16,)
    _tensor_checks(dev, (q, "q", bf, None), (k, "k", bf, (B, S, Hkv, D)),
                   (v, "v", bf, (B, S, Hkv, D)), (out, "out", bf, (B, S, H, D)),
                   (dout, "dout", bf, (B, S, H, D)), (lse, "lse", (torch.float32,), (B, H, S)),
                   (dq, "dq", bf, (B, S, H, D)), (dk, "dk", bf, (B, S, Hkv, D)),
                   (dv, "dv", bf, (B, S, Hkv, D)))
    if scale is None:
        scale = D ** -0.5
    code = _call_on(dev, stream, lambda sp: lib.ra_bwd_static(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
        dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, S, D, int(P),
        int(bool(causal)), float(scale), sp))
    _check(code, "ra_bwd_static")
    return dq, dk, dv


def ra_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, lse_ptr: int | None, B: int,
               H: int, Hkv: int, S: int, D: int, P: int, causal: bool, scale: float,
               stream=None) -> int:
    """The C call with plain integers (device addresses); returns the status code."""
    return int(_load().ra_fwd(q_ptr, k_ptr, v_ptr, out_ptr, lse_ptr, B, H, Hkv, S, D, P,
                              int(bool(causal)), float(scale), _stream_ptr(stream)))


def ra_merge_partials(o_parts, lse_parts, *, out=None, lse=None, want_lse: bool = True,
                      stream=None):
    """Merge ``n`` normalised partials: ``o_parts`` [n,B,S,H,D] (bf16 or
    fp32), ``lse_parts`` [n,B,H,S] fp32.  Returns ``(out, lse)``."""
    import torch

    lib = _load()
    n, B, S, H, D = _dims(o_parts, "o_parts", 5)
    dev = o_parts.device
    _tensor_checks(dev, (o_parts, "o_parts", (torch.bfloat16, torch.float32), None),
                   (lse_parts, "lse_parts", (torch.float32,), (n, B, H, S)))
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    _tensor_checks(dev, (out, "out", (torch.bfloat16,), (B, S, H, D)))
    if lse is not None:
        _tensor_checks(dev, (lse, "lse", (torch.float32,), (B, H, S)))
    code = _call_on(dev, stream, lambda sp: lib.ra_merge_partials(
        o_parts.data_ptr(), int(o_parts.dtype == torch.float32), lse_parts.data_ptr(), n,
        out.data_ptr(), None if lse is None else lse.data_ptr(), B, H, S, D, sp))
    _check(code, "ra_merge_partials")
    return out, lse


def ra_measure_ceilings(device=None) -> dict:
    """ex2 (MUFU) and fp32 FMA rates of a device, measured by the library's
    microbenchmark kernels (see include/ringattn.h)."""
    import torch

    lib = _load()
    out = (ctypes.c_double * 8)()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib.ra_measure_ceilings(out), "ra_measure_ceilings")
    keys = ("ex2_per_sm_clk", "ex2_per_s", "ffma_lanes_per_sm_clk", "ffma_lanes_per_s",
            "ffma2_lanes_per_sm_clk", "ffma2_lanes_per_s", "sm_mhz", "sms")
    return dict(zip(keys, list(out)))


def ra_get_last_device_status(stream=None) -> int:
    """Synchronise ``stream``, read and clear the device status word; returns
    the status code (``RA_OK`` or ``RA_ERR_TIMEOUT`` or ``RA_ERR_CUDA``)."""
    return int(_load().ra_get_last_device_status(_stream_ptr(stream)))


def ra_debug_set_fault(timeout_ns: int, skip_value_load: bool) -> None:
    _load().ra_debug_set_fault(int(timeout_ns), int(bool(skip_value_load)))


MMA_ORDER_STRICT, MMA_ORDER_GROUPED, MMA_ORDER_INORDER, MMA_ORDER_BRIDGED = 0, 1, 2, 3


def ra_set_mma_order(order: int) -> None:
    """MMA issue order of subsequent ra_fwd / ra_fwd_block launches:
    3 bridged by a tcgen05.shift (default), 0 strict (commit wait), 1 grouped,
    2 in-order with nothing between (for measurement only); see
    include/ringattn.h."""
    _load().ra_set_mma_order(int(order))


def ra_debug_build() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(_load().ra_debug_build() & 1)


def ra_trace_build() -> bool:
    """True when the loaded library is the traced build."""
    return bool(_load().ra_debug_build() & 2)


def ra_trace_read(n_ctas: int = 152):
    """Per-role cycle counters of the last forward launch (traced builds):
    an int64 tensor [n_ctas, 32]; see ring_chunked_attention_gb300.trace."""
    import torch

    buf = (ctypes.c_ulonglong * (32 * n_ctas))()
    _check(_load().ra_trace_read(buf, int(n_ctas)), "ra_trace_read")
    return torch.tensor(list(buf), dtype=torch.int64).view(n_ctas, 32)


def ra_debug_set_bounds_trim(elements: int) -> None:
    """Bounds-checked builds: the last ``elements`` elements of every checked
    buffer count as outside it (a test hook; 0 turns it off)."""
    _load().ra_debug_set_bounds_trim(int(elements))


def ra_set_item_pairing(policy: int) -> None:
    """0 automatic (default), 1 pair query tiles whenever possible, 2 never."""
    _load().ra_set_item_pairing(int(policy))


def ra_shutdown() -> None:
    _load().ra_shutdown()
