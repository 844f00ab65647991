"""GPU parity of the layer prologue and epilogue (include/gdn_layer.h) against
the fp64 layer oracle, through the C ABI.

Tolerances: bf16 outputs (q, k, v, o) max|gpu - oracle| / max|oracle| <= 1e-2
per tensor (one bf16 rounding of an fp32 result); alpha, beta (fp32) within
2e-6 absolute; convolution states (copies of bf16 inputs) bit-exact."""
import numpy as np
import pytest
import torch

from oracle import layer as OL
from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn
from linear_attention_recurrence_14_b300.inputs import make_layer_inputs

from .helpers import rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-2
GATE_TOL = 2e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()


def _prologue(x, state_out=True):
    return gdn.layer_prologue(x.xq, x.xk, x.xv, x.wq, x.wk, x.wv, x.a_raw, x.b_raw, x.A, x.b_alpha,
                              state_q=x.state_q, state_k=x.state_k, state_v=x.state_v, state_out=state_out)


def _oracle_prologue(x):
    return OL.prologue(x.xq, x.xk, x.xv, x.wq, x.wk, x.wv, x.a_raw, x.b_raw, x.A, x.b_alpha,
                       x.state_q, x.state_k, x.state_v)


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy()


@pytest.mark.parametrize(
    "B,T,Hqk,Hv,d,K,state",
    [
        (1, 1, 1, 2, 128, 4, True),      # one token: every tap but the current one from the state
        (1, 2, 1, 2, 128, 4, True),      # T < K - 1: the outgoing state mixes old state and inputs
        (2, 100, 2, 4, 128, 4, False),   # two tiles, ragged tail, zero state
        (1, 200, 1, 1, 64, 3, True),     # d = 64, three taps
        (1, 130, 2, 2, 128, 1, False),   # pointwise "convolution"
        (1, 257, 2, 4, 128, 2, True),    # tile boundaries at 64, 128, 192, 256
    ],
)
def test_prologue_matches_oracle(B, T, Hqk, Hv, d, K, state):
    x = make_layer_inputs(B, T, Hqk, Hv, d, K, seed=T + 7 * K, device="cuda", with_state=state, vary_heads=True)
    out = _prologue(x)
    ref = _oracle_prologue(x)
    for n in ("q", "k", "v"):
        assert rel_err(out[n], ref[n]) <= TOL, n
    for n in ("alpha", "beta"):
        assert np.max(np.abs(out[n].double().cpu().numpy() - ref[n])) <= GATE_TOL, n
    for n in ("state_q", "state_k", "state_v"):
        if K > 1:
            assert np.array_equal(_bits(out[n]), _bits(torch.tensor(ref[n]).to(torch.bfloat16))), n


def test_prologue_zero_tokens_copies_the_state():
    x = make_layer_inputs(1, 0, 1, 2, 128, 4, device="cuda", with_state=True)
    out = _prologue(x)
    for n in ("q", "k", "v"):
        assert torch.equal(out["state_" + n], getattr(x, "state_" + n))
    x = make_layer_inputs(1, 0, 1, 2, 128, 4, device="cuda", with_state=False)
    out = _prologue(x)
    assert not torch.any(out["state_v"].float() != 0)


def test_prologue_continuation_is_bit_exact():
    # one call over T tokens == two calls with the convolution state carried
    x = make_layer_inputs(1, 300, 2, 4, 128, 4, seed=5, device="cuda", with_state=True, vary_heads=True)
    full = _prologue(x)
    for cut in (1, 3, 64, 131):
        sl = lambda t, a, b: t[:, a:b].contiguous()  # noqa: E731
        first = gdn.layer_prologue(sl(x.xq, 0, cut), sl(x.xk, 0, cut), sl(x.xv, 0, cut), x.wq, x.wk, x.wv,
                                   sl(x.a_raw, 0, cut), sl(x.b_raw, 0, cut), x.A, x.b_alpha,
                                   state_q=x.state_q, state_k=x.state_k, state_v=x.state_v, state_out=True)
        second = gdn.layer_prologue(sl(x.xq, cut, 300), sl(x.xk, cut, 300), sl(x.xv, cut, 300), x.wq, x.wk, x.wv,
                                    sl(x.a_raw, cut, 300), sl(x.b_raw, cut, 300), x.A, x.b_alpha,
                                    state_q=first["state_q"], state_k=first["state_k"], state_v=first["state_v"],
                                    state_out=True)
        for n in ("q", "k", "v", "alpha", "beta"):
            assert torch.equal(torch.cat([first[n], second[n]], 1), full[n]), (cut, n)
        for n in ("state_q", "state_k", "state_v"):
            assert torch.equal(second[n], full[n]), (cut, n)


@pytest.mark.parametrize("B,T,Hv,d,eps", [(1, 100, 4, 128, 1e-6), (2, 33, 2, 64, 1e-6), (1, 1, 1, 128, 1e-3),
                                          (3, 77, 8, 128, 1e-6)])
def test_epilogue_matches_oracle(B, T, Hv, d, eps):
    x = make_layer_inputs(B, T, 1, Hv, d, seed=B * T + d, device="cuda")
    o = gdn.layer_epilogue(x.y, x.z, x.norm_w, eps)
    ref = OL.epilogue(x.y, x.z, x.norm_w, eps)
    assert rel_err(o, ref) <= TOL


def test_layer_full_size_windows_match_oracle():
    # B=1, Hqk=16, Hv=32, T=65536, d=128, K=4: the prologue and epilogue in the
    # configuration the benchmark times; sampled token windows (start, middle,
    # end) checked against the oracle started from the same convolution state.
    T = 65536
    x = make_layer_inputs(1, T, 16, 32, 128, 4, seed=0, device="cuda", with_state=True, vary_heads=True)
    out = _prologue(x)
    o = gdn.layer_epilogue(x.y, x.z, x.norm_w, 1e-6)
    for t0, t1 in ((0, 96), (T // 2 - 40, T // 2 + 40), (T - 96, T)):
        def win(t, a=t0, b=t1):
            return t[:, a:b]

        def state(name, H):
            if t0 == 0:
                return getattr(x, name)
            src = {"state_q": x.xq, "state_k": x.xk, "state_v": x.xv}[name]
            return src[:, t0 - 3:t0].reshape(1, 3, H * 128)
        ref = OL.prologue(win(x.xq), win(x.xk), win(x.xv), x.wq, x.wk, x.wv, win(x.a_raw), win(x.b_raw), x.A,
                          x.b_alpha, state("state_q", 16), state("state_k", 16), state("state_v", 32))
        for n in ("q", "k", "v"):
            assert rel_err(win(out[n]), ref[n]) <= TOL, (t0, n)
        for n in ("alpha", "beta"):
            assert np.max(np.abs(win(out[n]).double().cpu().numpy() - ref[n])) <= GATE_TOL, (t0, n)
        assert rel_err(win(o), OL.epilogue(win(x.y), win(x.z), x.norm_w)) <= TOL, t0
    assert np.array_equal(_bits(out["state_v"]), _bits(x.xv[:, T - 3:].reshape(1, 3, 32 * 128)))
