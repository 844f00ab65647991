"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/*.h declares, and rejects bad arguments on the host before any CUDA
call (the pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gdn.lib()


def declared_functions():
    text = "".join(open(os.path.join(ROOT, "include", h)).read()
                   for h in sorted(os.listdir(os.path.join(ROOT, "include"))) if h.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert set(names) == set(gdn.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    for code in range(9):
        assert L.gdn_status_string(code)
    assert L.gdn_status_string(1234) == b"unknown status"
    assert L.gdn_abi_version() == 10000


def shape(B=1, T=64, Hqk=2, Hv=4, d=128, dtype=gdn.GDN_BF16):
    return gdn.GdnShape(B, T, Hqk, Hv, d, d, dtype)


def test_workspace_bytes(L):
    s = shape(B=2, Hv=4, d=128)   # one chunk: status and staging only
    assert gdn.workspace_bytes(s) == 256 + 2 * 4 * 128 * 128 * 4
    # several chunks (bf16): the exact sequence split's segment flags and states, for at
    # most ceil(320 / (B * Hv)) segments (about two waves of a GPU of up to 160 SMs)
    r = lambda n: (n + 255) // 256 * 256  # noqa: E731
    s = shape(B=2, T=64 * 100, Hv=4, d=128)
    assert gdn.workspace_bytes(s) == r(256 + 8 * 128 * 128 * 4) + r(8 * 40 * 4) + 8 * 40 * 3 * 128 * 128 * 4
    s = shape(B=2, T=64 * 100, Hv=4, d=128, dtype=gdn.GDN_F32)
    assert gdn.workspace_bytes(s) == 256 + 8 * 128 * 128 * 4
    assert gdn.workspace_bytes(shape(Hqk=3, Hv=4)) == 0
    assert L.gdn_prefill_workspace_bytes(None) == 0


BASE = 1 << 32  # fake, 256-byte aligned device addresses; never dereferenced
MB = 1 << 20


def call_prefill(L, s, q=BASE, k=BASE + 64 * MB, v=BASE + 128 * MB, a=BASE + 192 * MB, b=BASE + 200 * MB,
                 S0=None, y=BASE + 256 * MB, S_T=BASE + 320 * MB, ws=BASE + 384 * MB, ws_bytes=None, opts=None):
    if ws_bytes is None:
        ws_bytes = max(gdn.workspace_bytes(s), 256) if s is not None else 256
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    o = None if opts is None else ctypes.byref(opts)
    return L.gdn_prefill_ex(ctypes.byref(s) if s is not None else None, o, vp(q), vp(k), vp(v), vp(a), vp(b),
                            vp(S0), vp(y), vp(S_T), vp(ws), ws_bytes, None)


def test_prefill_rejects_bad_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    assert call_prefill(L, None) == E["GDN_ERR_INVALID_ARG"]
    assert call_prefill(L, shape(Hqk=3, Hv=4)) == E["GDN_ERR_INVALID_ARG"]
    assert call_prefill(L, shape(T=-1)) == E["GDN_ERR_INVALID_ARG"]
    assert call_prefill(L, gdn.GdnShape(1, 64, 1, 1, 128, 128, 7)) == E["GDN_ERR_INVALID_ARG"]
    assert call_prefill(L, gdn.GdnShape(1, 64, 1, 1, 96, 96, 1)) == E["GDN_ERR_UNSUPPORTED"]
    assert call_prefill(L, gdn.GdnShape(1, 64, 1, 1, 128, 64, 1)) == E["GDN_ERR_UNSUPPORTED"]
    assert call_prefill(L, shape(), q=None) == E["GDN_ERR_INVALID_ARG"]
    assert call_prefill(L, shape(), ws=None) == E["GDN_ERR_WORKSPACE"]
    assert call_prefill(L, shape(), ws_bytes=255) == E["GDN_ERR_WORKSPACE"]
    assert call_prefill(L, shape(), q=BASE + 8) == E["GDN_ERR_ALIGNMENT"]
    assert call_prefill(L, shape(), a=BASE + 192 * MB + 2) == E["GDN_ERR_ALIGNMENT"]
    assert call_prefill(L, shape(), ws=BASE + 384 * MB + 16) == E["GDN_ERR_ALIGNMENT"]
    assert call_prefill(L, shape(), y=BASE) == E["GDN_ERR_ALIASING"]              # y == q
    assert call_prefill(L, shape(), S_T=BASE + 128 * MB) == E["GDN_ERR_ALIASING"]  # S_T inside v
    assert call_prefill(L, shape(), S0=BASE + 320 * MB + 256) == E["GDN_ERR_ALIASING"]  # partial S0/S_T overlap
    bad = gdn.GdnPrefillOptions(-1, 0.0, 0, 0)
    assert call_prefill(L, shape(), opts=bad) == E["GDN_ERR_INVALID_ARG"]
    bad = gdn.GdnPrefillOptions(0, 0.5, 0, 0)
    assert call_prefill(L, shape(), opts=bad) == E["GDN_ERR_INVALID_ARG"]
    bad = gdn.GdnPrefillOptions(0, 0.0, 0, 3)
    assert call_prefill(L, shape(), opts=bad) == E["GDN_ERR_INVALID_ARG"]
    bad = gdn.GdnPrefillOptions(0, 0.0, 0, 0, -1)
    assert call_prefill(L, shape(), opts=bad) == E["GDN_ERR_INVALID_ARG"]


def test_decode_rejects_bad_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    vp = ctypes.c_void_p
    s = shape(T=1)
    args = [vp(BASE), vp(BASE + MB), vp(BASE + 2 * MB), vp(BASE + 3 * MB), vp(BASE + 4 * MB), vp(BASE + 5 * MB),
            vp(BASE + 9 * MB)]
    assert L.gdn_decode_step(ctypes.byref(shape(T=2)), *args, None) == E["GDN_ERR_INVALID_ARG"]
    bad = list(args)
    bad[6] = vp(BASE + 5 * MB)  # y == S_inout
    assert L.gdn_decode_step(ctypes.byref(s), *bad, None) == E["GDN_ERR_ALIASING"]
    bad = list(args)
    bad[5] = None
    assert L.gdn_decode_step(ctypes.byref(s), *bad, None) == E["GDN_ERR_INVALID_ARG"]
    bad = list(args)
    bad[5] = vp(BASE + 5 * MB + 4)
    assert L.gdn_decode_step(ctypes.byref(s), *bad, None) == E["GDN_ERR_ALIGNMENT"]


def layer_shape(B=1, T=64, Hqk=2, Hv=4, d=128, K=4):
    return gdn.GdnLayerShape(B, T, Hqk, Hv, d, K)


def call_prologue(L, s, **over):
    names = [f[0] for f in gdn.GdnPrologueIO._fields_]
    vals = {n: BASE + i * 64 * MB for i, n in enumerate(names)}
    for n in ("state_q_in", "state_k_in", "state_v_in", "state_q_out", "state_k_out", "state_v_out"):
        vals[n] = None
    vals.update(over)
    io = gdn.GdnPrologueIO(*[vals[n] for n in names])
    return L.gdn_layer_prologue(ctypes.byref(s) if s is not None else None, ctypes.byref(io), None)


def test_layer_prologue_rejects_bad_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    assert call_prologue(L, None) == E["GDN_ERR_INVALID_ARG"]
    assert L.gdn_layer_prologue(ctypes.byref(layer_shape()), None, None) == E["GDN_ERR_INVALID_ARG"]
    assert call_prologue(L, layer_shape(Hqk=3, Hv=4)) == E["GDN_ERR_INVALID_ARG"]
    assert call_prologue(L, layer_shape(K=0)) == E["GDN_ERR_INVALID_ARG"]
    assert call_prologue(L, layer_shape(K=5)) == E["GDN_ERR_INVALID_ARG"]
    assert call_prologue(L, layer_shape(T=-1)) == E["GDN_ERR_INVALID_ARG"]
    assert call_prologue(L, layer_shape(d=96)) == E["GDN_ERR_UNSUPPORTED"]
    assert call_prologue(L, layer_shape(), xq=None) == E["GDN_ERR_INVALID_ARG"]
    assert call_prologue(L, layer_shape(), alpha=None) == E["GDN_ERR_INVALID_ARG"]
    assert call_prologue(L, layer_shape(), xv=BASE + 2 * 64 * MB + 8) == E["GDN_ERR_ALIGNMENT"]
    assert call_prologue(L, layer_shape(), A=BASE + 14 * 64 * MB + 2) == E["GDN_ERR_ALIGNMENT"]
    assert call_prologue(L, layer_shape(), state_v_out=BASE + 8) == E["GDN_ERR_ALIGNMENT"]
    # an output on top of an input, and two outputs on top of each other
    assert call_prologue(L, layer_shape(), q=BASE) == E["GDN_ERR_ALIASING"]
    assert call_prologue(L, layer_shape(), beta=BASE + 19 * 64 * MB) == E["GDN_ERR_ALIASING"]
    assert call_prologue(L, layer_shape(), state_q_in=BASE + 30 * 64 * MB,
                         state_q_out=BASE + 30 * 64 * MB) == E["GDN_ERR_ALIASING"]


def test_layer_epilogue_rejects_bad_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    vp = ctypes.c_void_p
    s = ctypes.byref(layer_shape())
    y, z, w, o = vp(BASE), vp(BASE + 64 * MB), vp(BASE + 128 * MB), vp(BASE + 192 * MB)
    assert L.gdn_layer_epilogue(None, y, z, w, 1e-6, o, None) == E["GDN_ERR_INVALID_ARG"]
    assert L.gdn_layer_epilogue(s, y, z, w, 0.0, o, None) == E["GDN_ERR_INVALID_ARG"]
    assert L.gdn_layer_epilogue(s, None, z, w, 1e-6, o, None) == E["GDN_ERR_INVALID_ARG"]
    assert L.gdn_layer_epilogue(s, vp(BASE + 8), z, w, 1e-6, o, None) == E["GDN_ERR_ALIGNMENT"]
    assert L.gdn_layer_epilogue(s, y, z, w, 1e-6, y, None) == E["GDN_ERR_ALIASING"]
    assert L.gdn_layer_epilogue(ctypes.byref(layer_shape(d=32)), y, z, w, 1e-6, o, None) == E["GDN_ERR_UNSUPPORTED"]


def test_host_prefill_workspace_and_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    s = shape(B=2, T=1000, Hqk=2, Hv=4, d=128)
    # pieces of 256 tokens: prefill workspace, two states, two slots of (q, k, v, y, alpha, beta)
    r = lambda n: (n + 255) // 256 * 256  # noqa: E731
    # gdn_prefill's workspace for one piece: status, staging, and the exact split's segment flags
    # and segment states (4 chunks: 4 segments x 8 heads x 3 states of 128 x 128 fp32)
    inner = r(r(256 + 2 * 4 * 128 * 128 * 4) + r(8 * 4 * 4) + 8 * 4 * 3 * 128 * 128 * 4)
    state = r(2 * 4 * 128 * 128 * 4)
    slot = 2 * r(2 * 256 * 2 * 128 * 2) + 2 * r(2 * 256 * 4 * 128 * 2) + 2 * r(2 * 256 * 4 * 4)
    assert gdn.host_workspace_bytes(s, 256) == inner + 2 * state + 2 * slot
    # default pieces: about T/8 tokens, a multiple of 64
    assert gdn.host_workspace_bytes(s, 0) == gdn.host_workspace_bytes(s, 128)
    assert gdn.host_workspace_bytes(s, -1) == 0
    assert gdn.host_workspace_bytes(shape(Hqk=3, Hv=4), 0) == 0
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    n = gdn.host_workspace_bytes(s, 256)

    def call(shp=s, tpp=256, q=BASE, ws=BASE + 512 * MB, ws_bytes=n):
        return L.gdn_prefill_host(ctypes.byref(shp), tpp, vp(q), vp(BASE + MB), vp(BASE + 2 * MB),
                                  vp(BASE + 3 * MB), vp(BASE + 4 * MB), None, vp(BASE + 5 * MB), None, vp(ws),
                                  ws_bytes, None)
    assert call(shp=shape(Hqk=3, Hv=4)) == E["GDN_ERR_INVALID_ARG"]
    assert call(shp=gdn.GdnShape(1, 64, 1, 1, 96, 96, 1)) == E["GDN_ERR_UNSUPPORTED"]
    assert call(tpp=-5) == E["GDN_ERR_INVALID_ARG"]
    assert call(ws=None) == E["GDN_ERR_WORKSPACE"]
    assert call(ws_bytes=n - 1) == E["GDN_ERR_WORKSPACE"]
    assert call(ws=BASE + 512 * MB + 16) == E["GDN_ERR_ALIGNMENT"]
    assert call(q=None) == E["GDN_ERR_INVALID_ARG"]


def test_channelwise_entry_points_reject_bad_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    s = ctypes.byref(shape(T=8))
    args = [vp(BASE), vp(BASE + MB), vp(BASE + 2 * MB), vp(BASE + 3 * MB), vp(BASE + 4 * MB)]
    assert L.gdn_prefill_cw(None, *args, None, vp(BASE + 5 * MB), vp(BASE + 6 * MB), None) == E["GDN_ERR_INVALID_ARG"]
    assert L.gdn_prefill_cw(s, None, *args[1:], None, vp(BASE + 5 * MB), vp(BASE + 6 * MB), None) == \
        E["GDN_ERR_INVALID_ARG"]
    assert L.gdn_prefill_cw(s, *args[:3], vp(BASE + 3 * MB + 4), args[4], None, vp(BASE + 5 * MB),
                            vp(BASE + 6 * MB), None) == E["GDN_ERR_ALIGNMENT"]
    assert L.gdn_prefill_cw(s, *args, None, vp(BASE), vp(BASE + 6 * MB), None) == E["GDN_ERR_ALIASING"]
    # decode: T must be 1
    assert L.gdn_decode_step_cw(s, *args, vp(BASE + 6 * MB), vp(BASE + 5 * MB), None) == E["GDN_ERR_INVALID_ARG"]


def test_backward_workspace_and_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    r = lambda n: (n + 255) // 256 * 256  # noqa: E731
    # checkpoints every 8 tokens, per-slab (32 value columns) partial sums of dq, dk, dbeta, dlog(alpha)
    for B, T, Hv, d in [(2, 1000, 4, 128), (1, 7, 2, 64), (3, 8, 2, 128)]:
        s = shape(B=B, T=T, Hqk=2, Hv=Hv, d=d)
        nc, ns = (T + 7) // 8, d // 32
        want = r(B * Hv * nc * d * d * 4) + 2 * r(B * T * Hv * ns * d * 4) + 2 * r(B * T * Hv * ns * 4)
        assert gdn.backward_workspace_bytes(s) == want
    assert gdn.backward_workspace_bytes(shape(T=0)) == 0
    assert gdn.backward_workspace_bytes(shape(Hqk=3, Hv=4)) == 0
    s = shape(B=1, T=64, Hqk=2, Hv=4, d=128)
    n = gdn.backward_workspace_bytes(s)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    # inputs at BASE + i*64MB (i = 0..7), outputs at BASE + (8 + i)*64MB, workspace at BASE + 16*64MB
    ins = dict(q=0, k=1, v=2, alpha=3, beta=4, S0=5, dy=6, dS_T=7)
    outs = dict(dq=8, dk=9, dv=10, dlog_alpha=11, dbeta=12, dS0=13)
    at = {**{k_: BASE + i * 64 * MB for k_, i in ins.items()}, **{k_: BASE + i * 64 * MB for k_, i in outs.items()}}

    def call(shp=s, ws=BASE + 16 * 64 * MB, ws_bytes=n, **over):
        a = {**at, **over}
        return L.gdn_backward(ctypes.byref(shp), *(vp(a[k_]) for k_ in ins), *(vp(a[k_]) for k_ in outs),
                              vp(ws), ws_bytes, None)
    assert call(shp=shape(Hqk=3, Hv=4)) == E["GDN_ERR_INVALID_ARG"]
    assert call(shp=gdn.GdnShape(1, 64, 1, 1, 96, 96, 1)) == E["GDN_ERR_UNSUPPORTED"]
    assert call(shp=gdn.GdnShape(1, 64, 1, 1 << 18, 128, 128, 1)) == E["GDN_ERR_UNSUPPORTED"]   # Hv * dk > 2^24
    for name in ("q", "dy", "dq", "dlog_alpha", "dbeta"):
        assert call(**{name: None}) == E["GDN_ERR_INVALID_ARG"], name
    assert call(ws=None) == E["GDN_ERR_WORKSPACE"]
    assert call(ws_bytes=n - 1) == E["GDN_ERR_WORKSPACE"]
    assert call(ws=BASE + 16 * 64 * MB + 16) == E["GDN_ERR_ALIGNMENT"]
    assert call(dy=at["dy"] + 8) == E["GDN_ERR_ALIGNMENT"]
    assert call(dv=at["dv"] + 4) == E["GDN_ERR_ALIGNMENT"]
    assert call(dbeta=at["dbeta"] + 2) == E["GDN_ERR_ALIGNMENT"]
    # an output on an input, two outputs on each other, the workspace on an output
    assert call(dq=at["q"]) == E["GDN_ERR_ALIASING"]
    assert call(dk=at["dq"] + 256) == E["GDN_ERR_ALIASING"]
    assert call(ws=at["dv"]) == E["GDN_ERR_ALIASING"]
    assert call(dS0=at["S0"]) == E["GDN_ERR_ALIASING"]
    # dS0 may be the very buffer of dS_T: past the host checks (no GPU here, so a CUDA/device status)
    assert call(dS0=at["dS_T"]) not in (E["GDN_ERR_ALIASING"], E["GDN_ERR_INVALID_ARG"], E["GDN_ERR_ALIGNMENT"])


def test_chunked_backward_workspace_and_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    r = lambda n: (n + 255) // 256 * 256  # noqa: E731
    # chunk records (74,240 bytes) and decay bounds (4 bytes) per (head, chunk); then the entering
    # states and the state gradients (bf16, 32 KB each per (head, chunk)); then dS0's staging
    # and the exact split's flags and segment maps (segs = min(chunks, ceil(320 / (B Hv))) per head)
    for B, T, Hv in [(2, 1000, 4), (1, 64, 2), (1, 65, 1)]:
        s = shape(B=B, T=T, Hqk=1, Hv=Hv, d=128)
        nc = (T + 63) // 64
        n = B * Hv * nc
        segs = min(nc, -(-320 // (B * Hv))) if nc > 1 else 0
        split = r(B * Hv * segs * 4) + B * Hv * segs * 3 * 128 * 128 * 4
        want = r(r(r(n * 74244) + 2 * n * 128 * 128 * 2) + split) + B * Hv * 128 * 128 * 4
        assert L.gdn_backward_chunked_workspace_bytes(ctypes.byref(s)) == want
    assert L.gdn_backward_chunked_workspace_bytes(ctypes.byref(shape(d=64))) == 0
    assert L.gdn_backward_chunked_workspace_bytes(ctypes.byref(shape(dtype=gdn.GDN_F32))) == 0
    s = shape(B=1, T=64, Hqk=2, Hv=4, d=128)
    n = L.gdn_backward_chunked_workspace_bytes(ctypes.byref(s))
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    names = ("q", "k", "v", "alpha", "beta", "S0", "dy", "dS_T", "dq", "dk", "dv", "dlog_alpha", "dbeta", "dS0")
    at = {k_: BASE + i * 64 * MB for i, k_ in enumerate(names)}

    def call(shp=s, ws=BASE + 16 * 64 * MB, ws_bytes=n, **over):
        a = {**at, **over}
        return L.gdn_backward_chunked(ctypes.byref(shp), *(vp(a[k_]) for k_ in names), vp(ws), ws_bytes, None)
    assert call(shp=shape(dtype=gdn.GDN_F32)) == E["GDN_ERR_UNSUPPORTED"]
    assert call(shp=shape(d=64)) == E["GDN_ERR_UNSUPPORTED"]
    assert call(shp=shape(Hqk=3, Hv=4)) == E["GDN_ERR_INVALID_ARG"]
    assert call(dy=None) == E["GDN_ERR_INVALID_ARG"]
    assert call(ws=None) == E["GDN_ERR_WORKSPACE"]
    assert call(ws_bytes=n - 1) == E["GDN_ERR_WORKSPACE"]
    assert call(dq=at["q"]) == E["GDN_ERR_ALIASING"]
    assert call(dv=at["dv"] + 4) == E["GDN_ERR_ALIGNMENT"]


def test_channelwise_chunked_workspace_and_arguments(L):
    E = {v: k for k, v in gdn.STATUS_NAMES.items()}
    r = lambda n: (n + 255) // 256 * 256  # noqa: E731
    for B, T, Hv in [(2, 1000, 4), (1, 1, 2)]:
        s = shape(B=B, T=T, Hqk=2, Hv=Hv, d=128)
        nc = (T + 63) // 64
        segs = min(nc, -(-320 // (B * Hv))) if nc > 1 else 0
        split = r(B * Hv * segs * 4) + r(B * Hv * segs * 3 * 128 * 128 * 4)
        want = r(256 + B * Hv * 128 * 128 * 4) + split + B * Hv * nc * 74244
        assert L.gdn_prefill_cw_workspace_bytes(ctypes.byref(s)) == want
    # shapes the token-sequential kernel takes need only the status area
    assert L.gdn_prefill_cw_workspace_bytes(ctypes.byref(shape(d=64))) == 256
    assert L.gdn_prefill_cw_workspace_bytes(ctypes.byref(shape(dtype=gdn.GDN_F32))) == 256
    s = shape(B=1, T=200, Hqk=2, Hv=4, d=128)
    n = L.gdn_prefill_cw_workspace_bytes(ctypes.byref(s))
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    names = ("q", "k", "v", "alpha", "beta", "S0", "y", "S_T")
    at = {k_: BASE + i * 64 * MB for i, k_ in enumerate(names)}

    def call(shp=s, opts=None, ws=BASE + 16 * 64 * MB, ws_bytes=n, **over):
        a = {**at, **over}
        return L.gdn_prefill_cw_ex(ctypes.byref(shp), None if opts is None else ctypes.byref(opts),
                                   *(vp(a[k_]) for k_ in names), vp(ws), ws_bytes, None)
    chunked = gdn.GdnPrefillOptions(0, 0.0, 0, gdn.ALGO_CHUNKED, 0)
    assert call(shp=shape(d=64), opts=chunked) == E["GDN_ERR_UNSUPPORTED"]
    assert call(opts=gdn.GdnPrefillOptions(-1, 0.0, 0, 0, 0)) == E["GDN_ERR_INVALID_ARG"]
    assert call(opts=gdn.GdnPrefillOptions(0, 0.0, 0, 0, 3)) == E["GDN_ERR_INVALID_ARG"]   # no stall hook here
    assert call(ws=None) == E["GDN_ERR_WORKSPACE"]
    assert call(ws_bytes=n - 1) == E["GDN_ERR_WORKSPACE"]
    assert call(ws=BASE + 16 * 64 * MB + 16) == E["GDN_ERR_ALIGNMENT"]
    assert call(alpha=at["alpha"] + 4) == E["GDN_ERR_ALIGNMENT"]   # 16-byte rows of the channel gate
    assert call(y=at["q"]) == E["GDN_ERR_ALIASING"]
    assert call(ws=at["y"]) == E["GDN_ERR_ALIASING"]
