"""Thin ctypes binding over ``libgdn.so`` (C ABI of ``include/gdn.h``).

Argument marshalling only: shapes are read from the tensors, raw device
pointers and the current CUDA stream are handed to the C entry points, and
every step of the computation runs in the library's kernels.  There is no
fallback: a missing library or a failed call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK = 0
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_ALIGNMENT",
                4: "GDN_ERR_WORKSPACE", 5: "GDN_ERR_CUDA", 6: "GDN_ERR_TIMEOUT", 7: "GDN_ERR_DEVICE",
                8: "GDN_ERR_ALIASING"}
GDN_F32, GDN_BF16 = 0, 1
ALGO_AUTO, ALGO_CHUNKED, ALGO_SEQUENTIAL = 0, 1, 2
ALGO_NAMES = {ALGO_AUTO: "auto", ALGO_CHUNKED: "chunked", ALGO_SEQUENTIAL: "sequential"}

# Every symbol include/gdn.h and include/gdn_layer.h declare.
EXPORTS = ("gdn_status_string", "gdn_prefill_workspace_bytes", "gdn_prefill", "gdn_prefill_ex",
           "gdn_decode_step", "gdn_read_device_status", "gdn_device_supported", "gdn_abi_version",
           "gdn_prefill_noalloc", "gdn_layer_prologue", "gdn_layer_epilogue", "gdn_prefill_host_workspace_bytes",
           "gdn_prefill_host", "gdn_prefill_cw", "gdn_decode_step_cw", "gdn_backward_workspace_bytes",
           "gdn_backward", "gdn_prefill_noalloc_status", "gdn_prefill_launches",
           "gdn_prefill_cw_workspace_bytes", "gdn_prefill_cw_ex", "gdn_backward_chunked_workspace_bytes",
           "gdn_backward_chunked")
NOALLOC_SCRATCH_BYTES = 256 + 8 * 1024 * 1024


class GdnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("Hqk", ctypes.c_int32), ("Hv", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class GdnPrefillOptions(ctypes.Structure):
    _fields_ = [("segments", ctypes.c_int32), ("log_eps", ctypes.c_float), ("max_warmup_chunks", ctypes.c_int32),
                ("algorithm", ctypes.c_int32), ("test_stall_chunk", ctypes.c_int32)]


class GdnLayerShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("Hqk", ctypes.c_int32), ("Hv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("kconv", ctypes.c_int32)]


class GdnPrologueIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "xq", "xk", "xv", "wq", "wk", "wv", "state_q_in", "state_k_in", "state_v_in",
        "state_q_out", "state_k_out", "state_v_out", "a_raw", "b_raw", "A", "b_alpha",
        "q", "k", "v", "alpha", "beta")]


class GdnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({_status_text(code)})")
        self.code = code


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load libgdn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with linear_attention_recurrence_14_b300.build")
            L = ctypes.CDLL(LIB_PATH)
            vp, fp, c_size = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t
            sp = ctypes.POINTER(GdnShape)
            L.gdn_status_string.restype = ctypes.c_char_p
            L.gdn_status_string.argtypes = [ctypes.c_int]
            L.gdn_prefill_workspace_bytes.restype = c_size
            L.gdn_prefill_workspace_bytes.argtypes = [sp]
            L.gdn_prefill_cw_workspace_bytes.restype = c_size
            L.gdn_prefill_cw_workspace_bytes.argtypes = [sp]
            L.gdn_prefill_cw_ex.restype = ctypes.c_int
            L.gdn_prefill_cw_ex.argtypes = [sp, ctypes.POINTER(GdnPrefillOptions), vp, vp, vp, fp, fp, fp, vp, fp, vp,
                                            c_size, vp]
            L.gdn_prefill_launches.restype = ctypes.c_int
            L.gdn_prefill_launches.argtypes = [sp, ctypes.POINTER(GdnPrefillOptions)]
            L.gdn_prefill.restype = ctypes.c_int
            L.gdn_prefill.argtypes = [sp, vp, vp, vp, fp, fp, fp, vp, fp, vp, c_size, vp]
            L.gdn_prefill_ex.restype = ctypes.c_int
            L.gdn_prefill_ex.argtypes = [sp, ctypes.POINTER(GdnPrefillOptions), vp, vp, vp, fp, fp, fp, vp, fp, vp,
                                         c_size, vp]
            L.gdn_prefill_noalloc.restype = ctypes.c_int
            L.gdn_prefill_noalloc.argtypes = [sp, vp, vp, vp, fp, fp, fp, vp, fp, vp]
            L.gdn_decode_step.restype = ctypes.c_int
            L.gdn_decode_step.argtypes = [sp, vp, vp, vp, fp, fp, fp, vp, vp]
            L.gdn_prefill_noalloc_status.restype = ctypes.c_int
            L.gdn_prefill_noalloc_status.argtypes = [vp]
            L.gdn_read_device_status.restype = ctypes.c_int
            L.gdn_read_device_status.argtypes = [vp, vp]
            L.gdn_layer_prologue.restype = ctypes.c_int
            L.gdn_layer_prologue.argtypes = [ctypes.POINTER(GdnLayerShape), ctypes.POINTER(GdnPrologueIO), vp]
            L.gdn_layer_epilogue.restype = ctypes.c_int
            L.gdn_layer_epilogue.argtypes = [ctypes.POINTER(GdnLayerShape), vp, vp, fp, ctypes.c_float, vp, vp]
            L.gdn_prefill_host_workspace_bytes.restype = c_size
            L.gdn_prefill_host_workspace_bytes.argtypes = [sp, ctypes.c_int64]
            L.gdn_prefill_host.restype = ctypes.c_int
            L.gdn_prefill_host.argtypes = [sp, ctypes.c_int64, vp, vp, vp, fp, fp, fp, vp, fp, vp, c_size, vp]
            L.gdn_prefill_cw.restype = ctypes.c_int
            L.gdn_prefill_cw.argtypes = [sp, vp, vp, vp, fp, fp, fp, vp, fp, vp]
            L.gdn_decode_step_cw.restype = ctypes.c_int
            L.gdn_decode_step_cw.argtypes = [sp, vp, vp, vp, fp, fp, fp, vp, vp]
            L.gdn_backward_workspace_bytes.restype = c_size
            L.gdn_backward_workspace_bytes.argtypes = [sp]
            L.gdn_backward.restype = ctypes.c_int
            L.gdn_backward.argtypes = [sp, vp, vp, vp, fp, fp, fp, vp, fp, fp, fp, fp, fp, fp, fp, vp, c_size, vp]
            L.gdn_backward_chunked_workspace_bytes.restype = c_size
            L.gdn_backward_chunked_workspace_bytes.argtypes = [sp]
            L.gdn_backward_chunked.restype = ctypes.c_int
            L.gdn_backward_chunked.argtypes = L.gdn_backward.argtypes
            L.gdn_device_supported.restype = ctypes.c_int
            L.gdn_abi_version.restype = ctypes.c_int
            _lib = L
    return _lib


def _status_text(code: int) -> str:
    try:
        return lib().gdn_status_string(code).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(code: int, what: str):
    if code != GDN_OK:
        raise GdnError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _require(tensors: dict):
    """The C ABI takes dense row-major device buffers: reject views it cannot address."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, expected {dev}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def shape_of(q: torch.Tensor, v: torch.Tensor) -> GdnShape:
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    return GdnShape(B, T, Hqk, Hv, dk, dv, _dtype_code(q))


def workspace_bytes(shape: GdnShape) -> int:
    return int(lib().gdn_prefill_workspace_bytes(ctypes.byref(shape)))


def new_workspace(shape: GdnShape, device) -> torch.Tensor:
    """A zeroed workspace of the size gdn_prefill needs (uint8, 256-byte aligned by the allocator)."""
    return torch.zeros(max(workspace_bytes(shape), 256), dtype=torch.uint8, device=device)


def prefill(q, k, v, alpha, beta, S0=None, *, y=None, S_T=None, workspace=None, segments=0, log_eps=0.0,
            max_warmup_chunks=0, algorithm=ALGO_AUTO, test_stall_chunk=0, stream=None):
    """Run gdn_prefill_ex on device tensors; returns (y, S_T).

    q, k [B,T,Hqk,d]; v [B,T,Hv,d]; alpha, beta [B,T,Hv] fp32; S0 [B,Hv,d,d] fp32 or None.
    """
    _require(dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, y=y, S_T=S_T, workspace=workspace))
    shape = shape_of(q, v)
    if y is None:
        y = torch.empty_like(v)
    if S_T is None:
        S_T = torch.empty((shape.B, shape.Hv, shape.dk, shape.dv), dtype=torch.float32, device=v.device)
    own_ws = workspace is None
    if own_ws:
        # The zero fill must precede the prefill on the stream it runs on.
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream(v.device)):
            workspace = new_workspace(shape, v.device)
    opts = GdnPrefillOptions(segments, log_eps, max_warmup_chunks, algorithm, test_stall_chunk)
    rc = lib().gdn_prefill_ex(ctypes.byref(shape), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                              _ptr(beta), _ptr(S0), _ptr(y), _ptr(S_T), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "gdn_prefill_ex")
    if own_ws and stream is not None:
        # allocated on the current stream but used on `stream`: keep it from being reused too early
        workspace.record_stream(stream)
    return y, S_T


def prefill_noalloc(q, k, v, alpha, beta, S0=None, *, y=None, S_T=None, stream=None):
    """Run gdn_prefill_noalloc (no workspace; the library's fixed scratch array); returns (y, S_T)."""
    _require(dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, y=y, S_T=S_T))
    shape = shape_of(q, v)
    if y is None:
        y = torch.empty_like(v)
    if S_T is None:
        S_T = torch.empty((shape.B, shape.Hv, shape.dk, shape.dv), dtype=torch.float32, device=v.device)
    rc = lib().gdn_prefill_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                   _ptr(S0), _ptr(y), _ptr(S_T), _stream(stream))
    _check(rc, "gdn_prefill_noalloc")
    return y, S_T


def noalloc_status(stream=None) -> int:
    """Synchronise and return (and clear) the device status the no-alloc calls recorded."""
    return int(lib().gdn_prefill_noalloc_status(_stream(stream)))


def decode_step(q, k, v, alpha, beta, S, *, y=None, stream=None):
    """Run gdn_decode_step: one token per sequence, S [B,Hv,d,d] fp32 updated in place; returns y."""
    _require(dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S=S, y=y))
    shape = shape_of(q, v)
    if y is None:
        y = torch.empty_like(v)
    rc = lib().gdn_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S),
                               _ptr(y), _stream(stream))
    _check(rc, "gdn_decode_step")
    return y


def layer_prologue(xq, xk, xv, wq, wk, wv, a_raw, b_raw, A, b_alpha, *, state_q=None, state_k=None,
                   state_v=None, state_out=False, out=None, stream=None):
    """Run gdn_layer_prologue: q, k, v (bf16) and alpha, beta (fp32) from the projected features.

    xq, xk [B,T,Hqk,d] and xv [B,T,Hv,d] bf16; wq, wk [Hqk*d, K], wv [Hv*d, K] fp32 taps;
    a_raw, b_raw [B,T,Hv] fp32; A, b_alpha [Hv] fp32; optional incoming convolution states
    [B, K-1, H*d] bf16.  Returns a dict with q, k, v, alpha, beta and, with state_out=True,
    the outgoing states state_q, state_k, state_v."""
    _require(dict(xq=xq, xk=xk, xv=xv, wq=wq, wk=wk, wv=wv, a_raw=a_raw, b_raw=b_raw, A=A, b_alpha=b_alpha,
                  state_q=state_q, state_k=state_k, state_v=state_v))
    B, T, Hqk, d = xq.shape
    Hv = xv.shape[2]
    K = wq.shape[1]
    shape = GdnLayerShape(B, T, Hqk, Hv, d, K)
    dev = xq.device
    o = dict(out or {})
    o.setdefault("q", torch.empty_like(xq))
    o.setdefault("k", torch.empty_like(xk))
    o.setdefault("v", torch.empty_like(xv))
    o.setdefault("alpha", torch.empty((B, T, Hv), dtype=torch.float32, device=dev))
    o.setdefault("beta", torch.empty((B, T, Hv), dtype=torch.float32, device=dev))
    if state_out:
        o.setdefault("state_q", torch.empty((B, K - 1, Hqk * d), dtype=torch.bfloat16, device=dev))
        o.setdefault("state_k", torch.empty((B, K - 1, Hqk * d), dtype=torch.bfloat16, device=dev))
        o.setdefault("state_v", torch.empty((B, K - 1, Hv * d), dtype=torch.bfloat16, device=dev))
    _require(o)
    io = GdnPrologueIO(*[None if t is None else t.data_ptr() for t in (
        xq, xk, xv, wq, wk, wv, state_q, state_k, state_v, o.get("state_q"), o.get("state_k"), o.get("state_v"),
        a_raw, b_raw, A, b_alpha, o["q"], o["k"], o["v"], o["alpha"], o["beta"])])
    rc = lib().gdn_layer_prologue(ctypes.byref(shape), ctypes.byref(io), _stream(stream))
    _check(rc, "gdn_layer_prologue")
    return o


def layer_epilogue(y, z, norm_w, eps=1e-6, *, o=None, Hqk=None, stream=None):
    """Run gdn_layer_epilogue: o = sigmoid(z) * RMSNorm(y) (zero-centred weight), bf16 [B,T,Hv,d]."""
    _require(dict(y=y, z=z, norm_w=norm_w, o=o))
    B, T, Hv, d = y.shape
    shape = GdnLayerShape(B, T, Hqk or Hv, Hv, d, 1)
    if o is None:
        o = torch.empty_like(y)
    rc = lib().gdn_layer_epilogue(ctypes.byref(shape), _ptr(y), _ptr(z), _ptr(norm_w), float(eps), _ptr(o),
                                  _stream(stream))
    _check(rc, "gdn_layer_epilogue")
    return o


def host_workspace_bytes(shape: GdnShape, tokens_per_piece: int = 0) -> int:
    return int(lib().gdn_prefill_host_workspace_bytes(ctypes.byref(shape), int(tokens_per_piece)))


def new_host_workspace(shape: GdnShape, device, tokens_per_piece: int = 0) -> torch.Tensor:
    """A zeroed device workspace for gdn_prefill_host."""
    n = host_workspace_bytes(shape, tokens_per_piece)
    if n == 0:
        raise ValueError("invalid shape for gdn_prefill_host")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def prefill_host(q, k, v, alpha, beta, S0=None, *, y=None, S_T=None, workspace=None, tokens_per_piece=0,
                 device=None, stream=None):
    """Run gdn_prefill_host on host (CPU, preferably pinned) tensors; returns (y, S_T) as host tensors.

    The copies overlap the prefill; the call returns once the work is queued on `stream`
    (default: the current stream of `device`), so synchronise before reading y and S_T."""
    for name, t in dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, y=y, S_T=S_T).items():
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous host tensor")
    shape = shape_of(q, v)
    if y is None:
        y = torch.empty_like(v).pin_memory()
    if S_T is None:
        S_T = torch.empty((shape.B, shape.Hv, shape.dk, shape.dv), dtype=torch.float32).pin_memory()
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = new_host_workspace(shape, device, tokens_per_piece)
    if stream is None:
        stream = torch.cuda.current_stream(device)
    rc = lib().gdn_prefill_host(ctypes.byref(shape), int(tokens_per_piece), _ptr(q), _ptr(k), _ptr(v),
                                _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(y), _ptr(S_T), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), ctypes.c_void_p(stream.cuda_stream))
    _check(rc, "gdn_prefill_host")
    # the work is still in flight: keep the device workspace from being reused before it ends
    workspace.record_stream(stream)
    return y, S_T


def prefill_cw(q, k, v, alpha, beta, S0=None, *, y=None, S_T=None, workspace=None, algorithm=ALGO_AUTO, segments=0,
               log_eps=0.0, max_warmup_chunks=0, stream=None):
    """Run gdn_prefill_cw_ex (channel-wise decay, alpha [B,T,Hv,dk] fp32); returns (y, S_T).
    bf16 with d = 128 takes the chunked tensor-core path, whose workspace is allocated here
    (on the call's stream) unless given."""
    _require(dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, y=y, S_T=S_T))
    shape = shape_of(q, v)
    if y is None:
        y = torch.empty_like(v)
    if S_T is None:
        S_T = torch.empty((shape.B, shape.Hv, shape.dk, shape.dv), dtype=torch.float32, device=v.device)
    own_ws = workspace is None
    if own_ws:
        workspace = new_cw_workspace(shape, v.device)
    opts = GdnPrefillOptions(segments, log_eps, max_warmup_chunks, algorithm, 0)
    rc = lib().gdn_prefill_cw_ex(ctypes.byref(shape), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                 _ptr(beta), _ptr(S0), _ptr(y), _ptr(S_T), _ptr(workspace), workspace.numel(),
                                 _stream(stream))
    _check(rc, "gdn_prefill_cw_ex")
    if own_ws and stream is not None:
        # allocated on the current stream but used on `stream`: keep it from being reused too early
        workspace.record_stream(stream)
    return y, S_T


def cw_workspace_bytes(shape: GdnShape) -> int:
    return int(lib().gdn_prefill_cw_workspace_bytes(ctypes.byref(shape)))


def new_cw_workspace(shape: GdnShape, device) -> torch.Tensor:
    """Workspace of gdn_prefill_cw_ex (uint8, 256-byte aligned by the allocator; every byte
    the chunked path reads it writes first, so it is not cleared)."""
    return torch.empty(max(cw_workspace_bytes(shape), 256), dtype=torch.uint8, device=device)


def decode_step_cw(q, k, v, alpha, beta, S, *, y=None, stream=None):
    """Run gdn_decode_step_cw (channel-wise decay, alpha [B,1,Hv,dk]): S updated in place; returns y."""
    _require(dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S=S, y=y))
    shape = shape_of(q, v)
    if y is None:
        y = torch.empty_like(v)
    rc = lib().gdn_decode_step_cw(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S),
                                  _ptr(y), _stream(stream))
    _check(rc, "gdn_decode_step_cw")
    return y


def backward_workspace_bytes(shape: GdnShape, chunked: bool = False) -> int:
    fn = lib().gdn_backward_chunked_workspace_bytes if chunked else lib().gdn_backward_workspace_bytes
    return int(fn(ctypes.byref(shape)))


def new_backward_workspace(shape: GdnShape, device, chunked: bool = False) -> torch.Tensor:
    """A workspace of the size gdn_backward (or gdn_backward_chunked) needs (uint8; no initialisation needed)."""
    return torch.empty(max(backward_workspace_bytes(shape, chunked), 256), dtype=torch.uint8, device=device)


def backward(q, k, v, alpha, beta, S0, dy, dS_T=None, *, dS0=True, out=None, workspace=None, stream=None,
             algorithm=ALGO_SEQUENTIAL):
    """Run gdn_backward (algorithm ALGO_SEQUENTIAL: fp32, token by token) or gdn_backward_chunked
    (ALGO_CHUNKED: tensor cores, bf16 with d = 128); returns a dict with dq, dk [B,T,Hqk,d],
    dv [B,T,Hv,d], dlog_alpha, dbeta [B,T,Hv] (fp32) and dS0 [B,Hv,d,d] (fp32; None when dS0=False).

    dlog_alpha is alpha * dL/dalpha.  dy has the dtype of q, k, v; dS_T (fp32) may be None (zero).
    out: optional dict of preallocated outputs with the same keys.
    """
    chunked = algorithm == ALGO_CHUNKED
    _require(dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, dy=dy, dS_T=dS_T, workspace=workspace))
    if dy.dtype != q.dtype:
        raise TypeError(f"dy is {dy.dtype}, expected {q.dtype}")
    shape = shape_of(q, v)
    B, T, Hqk, d = q.shape
    Hv = v.shape[2]
    dev = v.device
    o = dict(out or {})
    f32 = dict(dtype=torch.float32, device=dev)
    o.setdefault("dq", torch.empty((B, T, Hqk, d), **f32))
    o.setdefault("dk", torch.empty((B, T, Hqk, d), **f32))
    o.setdefault("dv", torch.empty((B, T, Hv, d), **f32))
    o.setdefault("dlog_alpha", torch.empty((B, T, Hv), **f32))
    o.setdefault("dbeta", torch.empty((B, T, Hv), **f32))
    if dS0 and "dS0" not in o:
        o["dS0"] = torch.empty((B, Hv, d, d), **f32)
    o.setdefault("dS0", None)
    _require(o)
    own_ws = workspace is None
    if own_ws:
        workspace = new_backward_workspace(shape, dev, chunked=chunked)
    fn = lib().gdn_backward_chunked if chunked else lib().gdn_backward
    rc = fn(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
            _ptr(dy), _ptr(dS_T), _ptr(o["dq"]), _ptr(o["dk"]), _ptr(o["dv"]), _ptr(o["dlog_alpha"]),
            _ptr(o["dbeta"]), _ptr(o["dS0"]), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "gdn_backward_chunked" if chunked else "gdn_backward")
    if own_ws and stream is not None:
        workspace.record_stream(stream)
    return o


def backward_launches(shape: GdnShape) -> int:
    """Kernel launches one gdn_backward call enqueues (the per-slab kernel and the reduction)."""
    return 2 if shape.B * shape.T * shape.Hv > 0 else 0


def prefill_launches(shape: GdnShape, algorithm=ALGO_AUTO, segments=0) -> int:
    """Kernels one gdn_prefill call enqueues for this shape with a full workspace
    (gdn_prefill_launches: 4 with the exact sequence split, else 1; 0 when empty)."""
    opts = GdnPrefillOptions(segments, 0.0, 0, algorithm, 0)
    n = lib().gdn_prefill_launches(ctypes.byref(shape), ctypes.byref(opts))
    if n < 0:
        raise GdnError(GDN_ERR_INVALID_ARG, "gdn_prefill_launches")
    return n


def read_device_status(workspace, stream=None) -> int:
    """Synchronise and return (and clear) the device status recorded in the workspace."""
    return int(lib().gdn_read_device_status(_ptr(workspace), _stream(stream)))
