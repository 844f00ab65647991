"""The allocation-free prefill entry point (gdn_prefill_noalloc), called
through the C ABI, against the workspace entry point (gdn_prefill).

This entry point exists for callers that cannot allocate device memory (an
embedding runtime, a plugin inside another process, a fixed memory budget):
it takes no workspace and keeps its scratch in a fixed array inside the
library.  The file is named to be collected last, so a run that stops at its
first failure has already run every other test; it also passes on its own in
a fresh process (the array's address is looked up on the first call)."""
import ctypes

import pytest
import torch

from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn
from linear_attention_recurrence_14_b300.inputs import make_prefill_inputs

from .helpers import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()


def _noalloc_abi(x, y, S_T):
    """gdn_prefill_noalloc through ctypes with raw device pointers."""
    shape = gdn.shape_of(x.q, x.v)
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = gdn.lib().gdn_prefill_noalloc(ctypes.byref(shape), vp(x.q), vp(x.k), vp(x.v), vp(x.alpha), vp(x.beta),
                                       vp(x.S0), vp(y), vp(S_T),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("dtype,d,T,G", [("bf16", 128, 1000, 2), ("bf16", 64, 300, 1), ("f32", 64, 200, 2)])
def test_noalloc_matches_workspace_entry_point_twice(dtype, d, T, G):
    x = make_prefill_inputs(1, T, 2, 2 * G, d, dtype, decay_scale=0.05, s0_std=0.02, seed=31 + d, device="cuda")
    y_ref, S_ref = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    tol = TOL[x.q.dtype]
    for _ in range(2):   # two calls in a row share the scratch array
        y = torch.full_like(x.v, float("nan"))
        S_T = torch.full_like(S_ref, float("nan"))
        assert _noalloc_abi(x, y, S_T) == gdn.GDN_OK
        torch.cuda.synchronize()
        assert rel_err(y, y_ref.double().cpu().numpy()) <= tol
        assert rel_err(S_T, S_ref.double().cpu().numpy()) <= tol
    # no device-side error recorded in the array's status area
    assert gdn.noalloc_status() == gdn.GDN_OK


def test_noalloc_in_place_state():
    # S_T == S0: the final states are staged in the scratch array.
    x = make_prefill_inputs(2, 700, 1, 2, 128, "bf16", decay_scale=0.05, s0_std=0.05, seed=37, device="cuda")
    y_ref, S_ref = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    for _ in range(2):
        S = x.S0.clone()
        y = torch.empty_like(x.v)
        x_in = make_prefill_inputs(2, 700, 1, 2, 128, "bf16", decay_scale=0.05, s0_std=0.05, seed=37, device="cuda")
        x_in.S0 = S
        assert _noalloc_abi(x_in, y, S) == gdn.GDN_OK
        torch.cuda.synchronize()
        assert rel_err(y, y_ref.double().cpu().numpy()) <= TOL[torch.bfloat16]
        assert rel_err(S, S_ref.double().cpu().numpy()) <= TOL[torch.bfloat16]


def test_noalloc_out_of_place_needs_no_staging():
    # 130 (batch, value head) pairs at d = 128: an in-place call would not fit the
    # staging area, but an out-of-place call uses only the status area.
    x = make_prefill_inputs(130, 70, 1, 1, 128, "bf16", decay_scale=0.05, s0_std=0.02, seed=47, device="cuda")
    y_ref, S_ref = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    y = torch.full_like(x.v, float("nan"))
    S_T = torch.full_like(S_ref, float("nan"))
    assert _noalloc_abi(x, y, S_T) == gdn.GDN_OK
    torch.cuda.synchronize()
    assert rel_err(y, y_ref.double().cpu().numpy()) <= TOL[torch.bfloat16]
    assert rel_err(S_T, S_ref.double().cpu().numpy()) <= TOL[torch.bfloat16]
    assert gdn.noalloc_status() == gdn.GDN_OK


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # In place (S_T == S0), 129 (batch, value head) pairs at d = 128 would need more
    # staging than the fixed array holds: refused on the host before anything is
    # enqueued (the pointers are never dereferenced).
    shape = gdn.GdnShape(129, 64, 1, 1, 128, 128, gdn.GDN_BF16)
    assert gdn.workspace_bytes(shape) > gdn.NOALLOC_SCRATCH_BYTES
    base = 1 << 32
    q, k, v, a, b, S, y = (ctypes.c_void_p(base + i * (1 << 24)) for i in range(7))
    rc = gdn.lib().gdn_prefill_noalloc(ctypes.byref(shape), q, k, v, a, b, S, y, S, None)
    assert rc == 4  # GDN_ERR_WORKSPACE
    # head dims the kernels do not implement: the shape check's own status
    shape = gdn.GdnShape(1, 64, 1, 1, 96, 96, gdn.GDN_BF16)
    assert gdn.lib().gdn_prefill_noalloc(ctypes.byref(shape), q, k, v, a, b, S, y, S, None) == 2  # GDN_ERR_UNSUPPORTED
