"""Pins of the fp64 layer oracle (oracle/layer.py) against facts the pages and
the mathematics fix, each chosen so that a plausible mistake fails it: a tap
order reversed, the state not carried, sigma(-x) for sigma(x), a missing
(1 + w), a norm over the wrong axis, softplus replaced by exp or relu."""
import math

import numpy as np
import pytest

from oracle import layer as L



def rng(seed=0):
    return np.random.default_rng(seed)


def test_conv_current_tap_is_identity_and_first_tap_is_a_shift():
    x = rng(1).standard_normal((2, 9, 5))
    w = np.zeros((5, 4))
    w[:, 3] = 1.0
    out, st = L.short_conv(x, w)
    assert np.array_equal(out, x)
    assert np.array_equal(st, x[:, -3:, :])
    w = np.zeros((5, 4))
    w[:, 0] = 1.0
    state = rng(2).standard_normal((2, 3, 5))
    out, _ = L.short_conv(x, w, state)
    # tap 0 reads the input K-1 = 3 tokens back: the state for t < 3
    assert np.array_equal(out[:, :3], state)
    assert np.array_equal(out[:, 3:], x[:, :-3])


def test_conv_impulse_response_is_the_reversed_taps():
    K, T, C = 4, 10, 3
    w = rng(3).standard_normal((C, K))
    x = np.zeros((1, T, C))
    x[0, 2, 1] = 1.0
    out, _ = L.short_conv(x, w)
    expect = np.zeros((1, T, C))
    for j in range(K):
        expect[0, 2 + j, 1] = w[1, K - 1 - j]
    assert np.array_equal(out, expect)


def test_conv_state_carries_across_a_split():
    x = rng(4).standard_normal((2, 13, 6))
    w = rng(5).standard_normal((6, 4))
    s0 = rng(6).standard_normal((2, 3, 6))
    full, st_full = L.short_conv(x, w, s0)
    for cut in (1, 2, 3, 7):
        a, st = L.short_conv(x[:, :cut], w, s0)
        b, st2 = L.short_conv(x[:, cut:], w, st)
        assert np.allclose(np.concatenate([a, b], 1), full, rtol=0, atol=1e-14)
        assert np.array_equal(st2, st_full)


def test_conv_brute_force_small():
    x = rng(7).standard_normal((1, 6, 2))
    w = rng(8).standard_normal((2, 3))
    out, _ = L.short_conv(x, w)
    for t in range(6):
        for c in range(2):
            acc = 0.0
            for i in range(3):
                tt = t - 2 + i
                acc += w[c, i] * (x[0, tt, c] if tt >= 0 else 0.0)
            assert abs(out[0, t, c] - acc) < 1e-15


def test_silu_closed_forms():
    assert L.silu(np.array([0.0]))[0] == 0.0
    # sigma(ln 3) = 3/4, so SiLU(ln 3) = (3/4) ln 3
    assert abs(L.silu(np.array([math.log(3.0)]))[0] - 0.75 * math.log(3.0)) < 1e-15
    u = rng(9).standard_normal(50) * 4
    # sigma(-u) = 1 - sigma(u)  =>  SiLU(-u) = SiLU(u) - u
    assert np.allclose(L.silu(-u), L.silu(u) - u, rtol=0, atol=1e-13)


def test_sigmoid_and_softplus_closed_forms():
    assert L.sigmoid(np.array([0.0]))[0] == 0.5
    assert abs(L.softplus(np.array([0.0]))[0] - math.log(2.0)) < 1e-16
    u = rng(10).standard_normal(50) * 30
    # softplus(u) - softplus(-u) = u, and softplus > relu
    assert np.allclose(L.softplus(u) - L.softplus(-u), u, rtol=0, atol=1e-12)
    assert np.all(L.softplus(u) >= np.maximum(u, 0))
    m = np.linspace(-5, 5, 21)
    assert np.all(L.softplus(m) > np.maximum(m, 0))


def test_gates_closed_forms():
    # A = 0, a + b_alpha = 0: alpha = exp(-softplus(0)) = 1/2 exactly; beta(0) = 1/2
    a, b = L.gates(np.zeros((1, 1, 2)), np.zeros((1, 1, 2)), np.zeros(2), np.zeros(2))
    assert np.allclose(a, 0.5, rtol=0, atol=1e-16) and np.all(b == 0.5)
    # A = ln 2 doubles the exponent: alpha = 1/4; the bias shifts the argument
    a, _ = L.gates(np.full((1, 1, 2), -1.0), np.zeros((1, 1, 2)), np.full(2, math.log(2.0)), np.ones(2))
    assert np.allclose(a, 0.25, rtol=0, atol=1e-15)
    # per-head A: head 1 with exp(A) = 3 gives alpha_0 ** 3
    a, _ = L.gates(np.full((1, 4, 2), 0.3), np.zeros((1, 4, 2)), np.array([0.0, math.log(3.0)]), np.zeros(2))
    assert np.allclose(a[..., 1], a[..., 0] ** 3, rtol=1e-14)
    # alpha in (0, 1), decreasing in a
    a, _ = L.gates(np.linspace(-8, 8, 33).reshape(1, 33, 1), np.zeros((1, 33, 1)), np.zeros(1), np.zeros(1))
    assert np.all((a > 0) & (a < 1)) and np.all(np.diff(a[0, :, 0]) < 0)


def test_l2norm_unit_rows_scale_invariance():
    u = rng(11).standard_normal((3, 4, 16))
    n = L.l2norm(u, eps=0.0)
    assert np.allclose(np.linalg.norm(n, axis=-1), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(L.l2norm(7.5 * u, eps=0.0), n, rtol=0, atol=1e-14)
    # normalised per row of the last axis, not over the whole tensor
    assert not np.allclose(n, u / np.linalg.norm(u), atol=1e-3)


def test_rmsnorm_zero_centred_closed_forms():
    w = rng(12).standard_normal(8) * 0.1
    y = np.full((1, 1, 8), -3.0)
    # a constant vector normalises to its sign, scaled by (1 + w)
    assert np.allclose(L.rmsnorm_zc(y, w, eps=0.0), -(1.0 + w), rtol=0, atol=1e-15)
    u = rng(13).standard_normal((2, 5, 8))
    r = L.rmsnorm_zc(u, np.zeros(8), eps=0.0)
    assert np.allclose(np.sqrt(np.mean(r * r, axis=-1)), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(L.rmsnorm_zc(4 * u, w, eps=0.0), L.rmsnorm_zc(u, w, eps=0.0), rtol=0, atol=1e-14)


def test_epilogue_gate_limits():
    y = rng(14).standard_normal((1, 3, 2, 8))
    w = rng(15).standard_normal(8) * 0.1
    o = L.epilogue(y, np.zeros_like(y), w)
    assert np.allclose(o, 0.5 * L.rmsnorm_zc(y, w), rtol=0, atol=1e-15)
    o = L.epilogue(y, np.full_like(y, 60.0), w)
    assert np.allclose(o, L.rmsnorm_zc(y, w), rtol=0, atol=1e-14)
    assert np.allclose(L.epilogue(y, np.full_like(y, -60.0), w), 0.0, atol=1e-20)


def test_prologue_features_brute_force_tiny():
    # q = L2Norm(SiLU(conv)), v = SiLU(conv), written out one element at a time
    B, T, H, d, K = 1, 5, 2, 4, 3
    r = rng(16)
    xq = r.standard_normal((B, T, H, d))
    wq = r.standard_normal((H * d, K))
    q, st = L.feature(xq, wq, None, True, eps=0.0)
    v, _ = L.feature(xq, wq, None, False)
    for t in range(T):
        for h in range(H):
            u = []
            for e in range(d):
                c = h * d + e
                acc = 0.0
                for i in range(K):
                    tt = t - (K - 1) + i
                    if tt >= 0:
                        acc += wq[c, i] * xq[0, tt, h, e]
                u.append(acc / (1.0 + math.exp(-acc)))
            nrm = math.sqrt(sum(x * x for x in u))
            for e in range(d):
                assert abs(v[0, t, h, e] - u[e]) < 1e-14
                assert abs(q[0, t, h, e] - u[e] / nrm) < 1e-14
    assert st.shape == (B, K - 1, H * d)


def test_prologue_whole_brute_force_tiny():
    # The whole prologue as the reading notes' "Feature parameterization" and
    # "Gating dynamics" write it, one element at a time with its own loops:
    # q = L2Norm(SiLU(conv_q)), k = L2Norm(SiLU(conv_k)), v = SiLU(conv_v) (no
    # norm), alpha = exp(-e^A softplus(a + b_alpha)), beta = sigma(b), each
    # convolution reading its own incoming state, and the three outgoing states
    # (the last K-1 inputs of each stream).  Every input is distinct, so a
    # swapped state, tap set, gate input or a normalised v fails it.
    B, T, Hqk, Hv, d, K = 2, 3, 1, 2, 4, 4          # T < K-1 + 1: the outgoing state mixes state and input
    r = rng(17)
    xq, xk = r.standard_normal((B, T, Hqk, d)), r.standard_normal((B, T, Hqk, d))
    xv = r.standard_normal((B, T, Hv, d))
    wq, wk, wv = r.standard_normal((Hqk * d, K)), r.standard_normal((Hqk * d, K)), r.standard_normal((Hv * d, K))
    sq, sk = r.standard_normal((B, K - 1, Hqk * d)), r.standard_normal((B, K - 1, Hqk * d))
    sv = r.standard_normal((B, K - 1, Hv * d))
    a_raw, b_raw = r.standard_normal((B, T, Hv)), r.standard_normal((B, T, Hv))
    A, b_alpha = r.standard_normal(Hv) * 0.5, r.standard_normal(Hv) * 0.5
    out = L.prologue(xq, xk, xv, wq, wk, wv, a_raw, b_raw, A, b_alpha, sq, sk, sv)

    def stream_value(x, w, st, b, t, h, e):
        # conv input at time tt: the carried state for tt < 0, else the projection
        c = h * d + e
        acc = 0.0
        for i in range(K):
            tt = t - (K - 1) + i
            val = st[b, K - 1 + tt, c] if tt < 0 else x[b, tt, h, e]
            acc += w[c, i] * val
        return acc / (1.0 + math.exp(-acc))

    for b in range(B):
        for t in range(T):
            for name, x, w, st, H, norm in (("q", xq, wq, sq, Hqk, True), ("k", xk, wk, sk, Hqk, True),
                                            ("v", xv, wv, sv, Hv, False)):
                for h in range(H):
                    u = [stream_value(x, w, st, b, t, h, e) for e in range(d)]
                    scale = 1.0 / math.sqrt(sum(z * z for z in u) + 1e-6) if norm else 1.0
                    for e in range(d):
                        assert abs(out[name][b, t, h, e] - u[e] * scale) < 1e-13, (name, b, t, h, e)
            for h in range(Hv):
                zz = a_raw[b, t, h] + b_alpha[h]
                sp = math.log1p(math.exp(zz))
                assert abs(out["alpha"][b, t, h] - math.exp(-math.exp(A[h]) * sp)) < 1e-14
                assert abs(out["beta"][b, t, h] - 1.0 / (1.0 + math.exp(-b_raw[b, t, h]))) < 1e-15
        # outgoing states: the last K-1 conv inputs, oldest first
        for name, x, st, H in (("state_q", xq, sq, Hqk), ("state_k", xk, sk, Hqk), ("state_v", xv, sv, Hv)):
            for j in range(K - 1):
                tt = T - (K - 1) + j
                for c in range(H * d):
                    want = st[b, K - 1 + tt, c] if tt < 0 else x[b, tt, c // d, c % d]
                    assert out[name][b, j, c] == want, (name, b, j, c)
