"""ctypes wrapper around the plain-C fp64 oracle (``gdn_oracle.c``).

Test infrastructure only: the library never imports this module.

``recurrence`` runs the four-line gated delta recurrence of the Qwen3.8-Next
reading notes (jianyuh.github.io, section 2.1 "Gated DeltaNet") on every
(batch, value-head) pair, in fp64, sequentially over tokens.  Inputs are upcast
exactly from their stored dtype (bf16 and fp32 values are exact in fp64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/libgdn_oracle.so``."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        for fn in (lib.gdn_oracle_recurrence, lib.gdn_oracle_recurrence_cw):
            fn.restype = ctypes.c_int
            fn.argtypes = [
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
            ]
        _lib = lib
    return _lib


def _f64(x):
    """Exact upcast of a numpy array or torch tensor to a contiguous float64 array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (any device / dtype)
        import torch

        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def recurrence(q, k, v, alpha, beta, S0=None, threads: int | None = None):
    """Run the recurrence on full tensors.

    q, k: [B, T, Hqk, dk]; v: [B, T, Hv, dv]; beta: [B, T, Hv]; alpha: [B, T, Hv]
    (scalar decay) or [B, T, Hv, dk] (channel-wise decay, S~ = diag(alpha_t) S);
    S0: [B, Hv, dk, dv] or None (zeros).  Returns (y [B,T,Hv,dv], S_T [B,Hv,dk,dv])
    as float64 numpy arrays.
    """
    q, k, v, alpha, beta, S0 = (_f64(t) for t in (q, k, v, alpha, beta, S0))
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    cw = alpha.ndim == 4
    if k.shape != q.shape or v.shape[:2] != (B, T) or beta.shape != (B, T, Hv):
        raise ValueError("inconsistent shapes")
    if alpha.shape != ((B, T, Hv, dk) if cw else (B, T, Hv)):
        raise ValueError("alpha shape")
    if S0 is not None and S0.shape != (B, Hv, dk, dv):
        raise ValueError("S0 shape")
    y = np.zeros((B, T, Hv, dv), dtype=np.float64)
    S_T = np.zeros((B, Hv, dk, dv), dtype=np.float64)
    nthreads = threads if threads is not None else (os.cpu_count() or 1)
    fn = _load().gdn_oracle_recurrence_cw if cw else _load().gdn_oracle_recurrence
    rc = fn(
        B, T, Hqk, Hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
        _ptr(y), _ptr(S_T), nthreads,
    )
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return y, S_T


def recurrence_head(q, k, v, alpha, beta, S0, b: int, hv: int, T: int | None = None):
    """Run the recurrence for one (batch, value-head) pair only.

    Slices the pair's inputs (value head ``hv`` reads key head ``hv // (Hv/Hqk)``)
    and optionally only the first ``T`` tokens.  Returns (y [T, dv], S_T [dk, dv]).
    """
    Hqk, Hv = q.shape[2], v.shape[2]
    hk = hv // (Hv // Hqk)
    T = q.shape[1] if T is None else T
    sl = lambda x: x[b:b + 1, :T]  # noqa: E731
    qh = sl(q)[:, :, hk:hk + 1]
    kh = sl(k)[:, :, hk:hk + 1]
    vh = sl(v)[:, :, hv:hv + 1]
    ah = sl(alpha)[:, :, hv:hv + 1]
    bh = sl(beta)[:, :, hv:hv + 1]
    s0 = None if S0 is None else S0[b:b + 1, hv:hv + 1]
    y, st = recurrence(qh, kh, vh, ah, bh, s0, threads=1)
    return y[0, :, 0], st[0, 0]
