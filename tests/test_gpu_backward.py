"""GPU parity of the backward pass (gdn_backward) against the fp64 backward
oracle, through the C ABI.  The kernel computes in fp32 from inputs the oracle
also sees (bf16 inputs are exact in fp64), so both input dtypes take the fp32
tolerance 1e-4 on max|gpu - oracle| / max|oracle| per tensor; the same
algorithm run in numpy fp32 stays near 1e-6 on these shapes.  The decay
gradient is compared in log space: dlog_alpha = alpha * dL/dalpha."""
import numpy as np
import pytest
import torch

import oracle
import oracle.backward as obw
from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn
from linear_attention_recurrence_14_b300.inputs import make_backward_grads, make_prefill_inputs, workload_inputs

from .helpers import rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _reference(x, g):
    o = obw.recurrence_grad(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T)
    o["dlog_alpha"] = x.alpha.double().cpu().numpy() * o["dalpha"]
    return o


def _check(out, ref, names=("dq", "dk", "dv", "dlog_alpha", "dbeta", "dS0")):
    for n in names:
        assert rel_err(out[n], ref[n]) <= TOL, (n, rel_err(out[n], ref[n]))


@pytest.mark.parametrize("B,T,Hqk,Hv,d,dtype,s0,ds", [
    (1, 37, 1, 2, 128, "f32", 0.05, 1.0),     # grouped heads, ragged last chunk
    (2, 64, 2, 2, 64, "f32", 0.0, 1.0),      # whole chunks, zero initial state
    (1, 150, 1, 1, 128, "bf16", 0.02, 0.0),  # no state gradient
    (1, 5, 1, 2, 64, "bf16", 0.05, 1.0),     # shorter than one chunk
    (1, 9, 2, 4, 128, "bf16", 0.0, 0.5),     # one token past a chunk
    (3, 1, 1, 1, 64, "f32", 0.05, 1.0),      # a single token
])
def test_backward_matches_oracle(B, T, Hqk, Hv, d, dtype, s0, ds):
    x = make_prefill_inputs(B, T, Hqk, Hv, d, dtype, decay_scale=0.1, s0_std=s0, seed=T + d, device="cuda")
    g = make_backward_grads(B, T, Hv, d, dtype, ds_std=ds, seed=T + d, device="cuda")
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T)
    torch.cuda.synchronize()
    _check(out, _reference(x, g))


def test_backward_empty_sequence_and_in_place_state_gradient():
    x = make_prefill_inputs(2, 0, 1, 2, 64, "f32", s0_std=0.05, seed=1, device="cuda")
    g = make_backward_grads(2, 0, 2, 64, "f32", ds_std=1.0, seed=1, device="cuda")
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T)
    torch.cuda.synchronize()
    assert torch.equal(out["dS0"], g.dS_T)
    # dS0 written over dS_T
    x = make_prefill_inputs(1, 40, 1, 2, 128, "bf16", s0_std=0.02, seed=2, device="cuda")
    g = make_backward_grads(1, 40, 2, 128, "bf16", ds_std=1.0, seed=2, device="cuda")
    ref = _reference(x, g)
    dST = g.dS_T.clone()
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, dST, out={"dS0": dST})
    torch.cuda.synchronize()
    _check(out, ref)


def test_backward_is_deterministic_and_satisfies_linearity_identities():
    x = make_prefill_inputs(1, 100, 2, 4, 128, "bf16", s0_std=0.02, seed=3, device="cuda")
    g = make_backward_grads(1, 100, 4, 128, "bf16", ds_std=1.0, seed=3, device="cuda")
    a = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T)
    b = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T)
    torch.cuda.synchronize()
    for n in a:
        assert torch.equal(a[n], b[n]), n
    # (y, S_T) is linear in (v, S0) jointly and y is linear in q, so for L = <dy, y> + <dS_T, S_T>:
    # <dv, v> + <dS0, S0> = L and <dq, q> = <dy, y> (Euler's theorem for degree-one maps).
    y, S_T = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    ydy = float((g.dy.double().cpu().numpy() * y).sum())
    L = ydy + float((g.dS_T.double().cpu().numpy() * S_T).sum())
    lhs = float((a["dv"].double() * x.v.double()).sum() + (a["dS0"].double() * x.S0.double()).sum())
    assert abs(lhs - L) <= 1e-4 * max(1.0, abs(L))
    assert abs(float((a["dq"].double() * x.q.double()).sum()) - ydy) <= 1e-4 * max(1.0, abs(ydy))


def test_backward_training_shape_sampled_heads():
    # B=2, H=16, T=4096, d=128, bf16: the whole shape runs; eight (batch, head) pairs
    # spread over both sequences, including the first and the last head, are checked
    # against the oracle.
    x = workload_inputs("train", seed=0, device="cuda")
    g = make_backward_grads(2, 4096, 16, 128, "bf16", ds_std=1.0, seed=0, device="cuda")
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T)
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dS0"):
        assert torch.isfinite(out[n]).all(), n
    for b, heads in ((0, [0, 5, 10, 15]), (1, [2, 7, 12, 15])):
        sl = lambda t: t[b:b + 1, :, heads].contiguous()  # noqa: E731
        ref = obw.recurrence_grad(sl(x.q), sl(x.k), sl(x.v), sl(x.alpha), sl(x.beta), None, sl(g.dy),
                                  g.dS_T[b:b + 1, heads])
        ref["dlog_alpha"] = sl(x.alpha).double().cpu().numpy() * ref["dalpha"]
        got = {n: sl(out[n]) for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta")}
        got["dS0"] = out["dS0"][b:b + 1, heads]
        _check(got, ref)


# ----------------------------------------------------------------------------
# The chunked backward on the tensor cores (bf16, d = 128): bf16 operands with
# fp32 accumulation, so the bf16 tolerance of the forward (2e-2) applies.
CHUNKED_TOL = 2e-2


def _check_chunked(out, ref, names=("dq", "dk", "dv", "dlog_alpha", "dbeta", "dS0")):
    for n in names:
        assert rel_err(out[n], ref[n]) <= CHUNKED_TOL, (n, rel_err(out[n], ref[n]))


@pytest.mark.parametrize("B,T,Hqk,Hv,s0,ds,decay", [
    (1, 64, 1, 1, 0.02, 1.0, 0.1),       # one whole chunk
    (1, 37, 1, 2, 0.05, 1.0, 0.1),       # grouped heads, shorter than a chunk
    (2, 200, 2, 4, 0.0, 1.0, 0.1),       # several chunks, ragged tail, no initial state
    (1, 150, 1, 1, 0.02, 0.0, 0.5),      # strong decay, no state gradient
    (1, 1, 1, 2, 0.05, 1.0, 0.1),        # a single token
    (2, 333, 1, 4, 0.02, 1.0, 0.1),      # four value heads per key head (dq, dk summed by atomics)
])
def test_backward_chunked_matches_oracle(B, T, Hqk, Hv, s0, ds, decay):
    x = make_prefill_inputs(B, T, Hqk, Hv, 128, "bf16", decay_scale=decay, s0_std=s0, seed=T + 91, device="cuda")
    g = make_backward_grads(B, T, Hv, 128, "bf16", ds_std=ds, seed=T + 91, device="cuda")
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T, algorithm=gdn.ALGO_CHUNKED)
    torch.cuda.synchronize()
    _check_chunked(out, _reference(x, g))


def test_backward_chunked_segments_and_in_place_state_gradient():
    # 2000 tokens over 2 heads: the state chains split into segments with warm-up windows.
    x = make_prefill_inputs(1, 2000, 1, 2, 128, "bf16", decay_scale=0.1, s0_std=0.02, seed=93, device="cuda")
    g = make_backward_grads(1, 2000, 2, 128, "bf16", ds_std=1.0, seed=93, device="cuda")
    ref = _reference(x, g)
    dST = g.dS_T.clone()
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, dST, out={"dS0": dST},
                       algorithm=gdn.ALGO_CHUNKED)
    torch.cuda.synchronize()
    _check_chunked(out, ref)
    # agrees with the fp32 token-sequential backward
    seq = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T)
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
        assert rel_err(out[n], seq[n].double().cpu().numpy()) <= CHUNKED_TOL, n


def test_backward_chunked_training_shape_sampled_heads():
    # B=2, H=16, T=4096, d=128, bf16: eight (batch, head) pairs including the last head.
    x = workload_inputs("train", seed=0, device="cuda")
    g = make_backward_grads(2, 4096, 16, 128, "bf16", ds_std=1.0, seed=0, device="cuda")
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T, algorithm=gdn.ALGO_CHUNKED)
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dS0"):
        assert torch.isfinite(out[n]).all(), n
    for b, heads in ((0, [0, 5, 10, 15]), (1, [2, 7, 12, 15])):
        sl = lambda t: t[b:b + 1, :, heads].contiguous()  # noqa: E731
        ref = obw.recurrence_grad(sl(x.q), sl(x.k), sl(x.v), sl(x.alpha), sl(x.beta), None, sl(g.dy),
                                  g.dS_T[b:b + 1, heads])
        ref["dlog_alpha"] = sl(x.alpha).double().cpu().numpy() * ref["dalpha"]
        got = {n: sl(out[n]) for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta")}
        got["dS0"] = out["dS0"][b:b + 1, heads]
        _check_chunked(got, ref)


@pytest.mark.parametrize("decay", [0.0, 1.2e-4])   # alpha = 1 and alpha ~ 1 - 1e-4
def test_backward_chunked_exact_split_for_gates_that_do_not_decay(decay):
    # Over 256 chunks without any window, both state chains take the exact split; the result
    # must agree with the fp32 token-sequential backward (itself pinned to the oracle).
    T = 64 * 260 + 5
    x = make_prefill_inputs(1, T, 1, 2, 128, "bf16", decay_scale=decay, s0_std=0.02, seed=97, device="cuda")
    g = make_backward_grads(1, T, 2, 128, "bf16", ds_std=1.0, seed=97, device="cuda")
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T, algorithm=gdn.ALGO_CHUNKED)
    seq = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T)
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dS0"):
        assert rel_err(out[n], seq[n].double().cpu().numpy()) <= CHUNKED_TOL, n
