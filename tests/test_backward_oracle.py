"""Pins of the fp64 backward oracle (oracle/backward.py): central finite
differences of the pinned forward oracle, closed forms at special gates, and
planted mistakes that the pins must reject."""
import importlib.util

import numpy as np
import pytest

import oracle
import oracle.backward as BW

EPS = 1e-6


def _inputs(B, T, Hqk, Hv, dk, dv, seed):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, Hqk, dk))
    k = r.standard_normal((B, T, Hqk, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, Hv, dv))
    a = r.uniform(0.6, 1.0, (B, T, Hv))
    b = r.uniform(0.1, 0.9, (B, T, Hv))
    S0 = 0.5 * r.standard_normal((B, Hv, dk, dv))
    dy = r.standard_normal((B, T, Hv, dv))
    dST = r.standard_normal((B, Hv, dk, dv))
    return dict(q=q, k=k, v=v, alpha=a, beta=b, S0=S0), dy, dST


def _loss(inp, dy, dST):
    y, S_T = oracle.recurrence(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["S0"], threads=1)
    return float(np.sum(y * dy) + np.sum(S_T * dST))


@pytest.mark.parametrize("shape", [(1, 5, 1, 1, 3, 2), (1, 4, 1, 2, 3, 3), (2, 3, 2, 4, 2, 3)])
def test_backward_matches_central_differences(shape, bw=None):
    bw = bw or BW
    inp, dy, dST = _inputs(*shape, seed=sum(shape))
    g = bw.recurrence_grad(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["S0"], dy, dST)
    names = {"q": "dq", "k": "dk", "v": "dv", "alpha": "dalpha", "beta": "dbeta", "S0": "dS0"}
    for n, gn in names.items():
        x = inp[n]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + EPS
            lp = _loss(inp, dy, dST)
            x[idx] = old - EPS
            lm = _loss(inp, dy, dST)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * EPS)
        scale = max(1.0, float(np.abs(fd).max()))
        assert np.abs(g[gn] - fd).max() <= 1e-6 * scale, n


def test_backward_forward_outputs_match_oracle():
    inp, dy, dST = _inputs(1, 6, 1, 2, 4, 3, seed=7)
    g = BW.recurrence_grad(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["S0"], dy, dST)
    y, S_T = oracle.recurrence(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["S0"], threads=1)
    assert np.allclose(g["y"], y, rtol=0, atol=1e-13) and np.allclose(g["S_T"], S_T, rtol=0, atol=1e-13)


def test_backward_identity_gates_closed_form():
    # alpha = 1, beta = 0: S_t = S0, y_t = S0^T q_t, so dS0 = dS_T + sum_t q_t dy_t^T,
    # dq_t = S0 dy_t, dv = dk = 0, dalpha_t = <G_t, S0>, dbeta_t = k_t^T G_t e_t
    inp, dy, dST = _inputs(1, 5, 1, 1, 3, 2, seed=8)
    inp["alpha"][:] = 1.0
    inp["beta"][:] = 0.0
    g = BW.recurrence_grad(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["S0"], dy, dST)
    S0 = inp["S0"][0, 0]
    q, k, v = inp["q"][0, :, 0], inp["k"][0, :, 0], inp["v"][0, :, 0]
    assert np.allclose(g["dS0"][0, 0], dST[0, 0] + q.T @ dy[0, :, 0], rtol=0, atol=1e-12)
    assert np.allclose(g["dq"][0, :, 0], dy[0, :, 0] @ S0.T, rtol=0, atol=1e-12)
    assert np.abs(g["dv"]).max() == 0.0 and np.abs(g["dk"]).max() == 0.0
    for t in range(5):
        G = dST[0, 0] + q[t:].T @ dy[0, t:, 0]       # dL/dS_t
        e = v[t] - S0.T @ k[t]
        assert abs(g["dalpha"][0, t, 0] - np.sum(G * S0)) < 1e-12
        assert abs(g["dbeta"][0, t, 0] - k[t] @ G @ e) < 1e-12


MUTATIONS = {
    "output_term_dropped": ("G = G + np.outer(qt, dy[b, t, h])", "G = G + 0.0 * np.outer(qt, dy[b, t, h])"),
    "missing_residual_path": ("out[\"dk\"][b, t, hk] -= St @ de", "out[\"dk\"][b, t, hk] -= 0.0 * St @ de"),
    "wrong_sign_erase": ("Gt -= np.outer(kt, de)", "Gt += np.outer(kt, de)"),
    "decay_not_propagated": ("G = a * Gt", "G = Gt"),
    "dq_from_previous_state": ("out[\"dq\"][b, t, hk] += S @ dy[b, t, h]", "out[\"dq\"][b, t, hk] += Sp @ dy[b, t, h]"),
    "beta_dropped_in_de": ("de = bt * (G.T @ kt)", "de = G.T @ kt"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_backward_pins_reject_mutation(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(BW.__file__).read()
    assert before in src, name
    path = tmp_path / "bw_mut.py"
    path.write_text(src.replace(before, after))
    spec = importlib.util.spec_from_file_location("bw_mut", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with pytest.raises(AssertionError):
        test_backward_matches_central_differences((1, 4, 1, 2, 3, 3), bw=mod)


def test_backward_linearity_identities():
    # (y, S_T) is linear in (v, S0) jointly and y is linear in q, so for L = <dy, y> + <dS_T, S_T>:
    # <dv, v> + <dS0, S0> = L and <dq, q> = <dy, y>.
    inp, dy, dST = _inputs(2, 11, 1, 2, 5, 4, seed=21)
    g = BW.recurrence_grad(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["S0"], dy, dST)
    ydy = np.sum(g["y"] * dy)
    L = ydy + np.sum(g["S_T"] * dST)
    assert abs(np.sum(g["dv"] * inp["v"]) + np.sum(g["dS0"] * inp["S0"]) - L) < 1e-11 * max(1, abs(L))
    assert abs(np.sum(g["dq"] * inp["q"]) - ydy) < 1e-11 * max(1, abs(ydy))
