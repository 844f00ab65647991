"""Pins of the oracle's channel-wise decay mode (alpha per key channel,
S~ = diag(alpha_t) S): a closed form, brute force over explicit transition
matrices, and the reduction to the scalar gate.  A planted mistake (decay
applied per column instead of per row) must fail them."""
import ctypes
import subprocess

import numpy as np
import pytest

import oracle
import oracle.oracle as ormod


def _inputs(B, T, Hqk, Hv, dk, dv, seed, unit=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, Hqk, dk))
    k = r.standard_normal((B, T, Hqk, dk))
    if unit:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, Hv, dv))
    a = r.uniform(0.5, 1.0, (B, T, Hv, dk))
    b = r.uniform(0.0, 1.0, (B, T, Hv))
    S0 = r.standard_normal((B, Hv, dk, dv)) * 0.3
    return q, k, v, a, b, S0


def test_cw_beta_zero_is_per_channel_decay():
    q, k, v, a, b, S0 = _inputs(1, 7, 1, 2, 5, 3, seed=1)
    b[:] = 0.0
    y, S_T = oracle.recurrence(q, k, v, a, b, S0)
    for h in range(2):
        prod = np.ones(5)
        for t in range(7):
            prod = prod * a[0, t, h]
            S_t = prod[:, None] * S0[0, h]
            assert np.allclose(y[0, t, h], S_t.T @ q[0, t, 0], rtol=0, atol=1e-12)
        assert np.allclose(S_T[0, h], S_t, rtol=0, atol=1e-12)


@pytest.mark.parametrize("unit", [True, False])
def test_cw_transition_matrix_bruteforce(unit):
    # S_t = (I - beta_t k_t k_t^T) diag(alpha_t) S_{t-1} + beta_t k_t v_t^T, formed explicitly
    B, T, Hqk, Hv, dk, dv = 1, 9, 1, 2, 4, 6
    q, k, v, a, b, S0 = _inputs(B, T, Hqk, Hv, dk, dv, seed=2, unit=unit)
    y, S_T = oracle.recurrence(q, k, v, a, b, S0)
    for h in range(Hv):
        S = S0[0, h].copy()
        for t in range(T):
            kt = k[0, t, 0]
            M = (np.eye(dk) - b[0, t, h] * np.outer(kt, kt)) @ np.diag(a[0, t, h])
            S = M @ S + b[0, t, h] * np.outer(kt, v[0, t, h])
            assert np.allclose(y[0, t, h], S.T @ q[0, t, 0], rtol=0, atol=1e-12)
        assert np.allclose(S_T[0, h], S, rtol=0, atol=1e-12)


def test_cw_uniform_channels_equal_scalar_gate():
    q, k, v, a, b, S0 = _inputs(2, 11, 1, 2, 8, 8, seed=3)
    a_scalar = a[..., 0]
    a_uniform = np.repeat(a_scalar[..., None], 8, axis=-1)
    y1, S1 = oracle.recurrence(q, k, v, a_uniform, b, S0)
    y2, S2 = oracle.recurrence(q, k, v, a_scalar, b, S0)
    assert np.allclose(y1, y2, rtol=0, atol=1e-13) and np.allclose(S1, S2, rtol=0, atol=1e-13)


def test_cw_pins_reject_column_decay(tmp_path, monkeypatch):
    src = open(ormod._SRC).read()
    before = "                row[j] *= a;"
    assert before in src
    msrc = tmp_path / "cw_mut.c"
    msrc.write_text(src.replace(before, "                row[j] *= J->alpha_cw ? at[j % dk] : a;"))
    mlib = tmp_path / "libcwmut.so"
    subprocess.run(["gcc", "-O1", "-shared", "-fPIC", "-pthread", "-o", str(mlib), str(msrc)], check=True)
    lib = ctypes.CDLL(str(mlib))
    dp = ctypes.POINTER(ctypes.c_double)
    for fn in (lib.gdn_oracle_recurrence, lib.gdn_oracle_recurrence_cw):
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_int64, ctypes.c_int64] + [ctypes.c_int] * 4 + [dp] * 8 + [ctypes.c_int]
    monkeypatch.setattr(ormod, "_lib", lib)
    with pytest.raises(AssertionError):
        test_cw_transition_matrix_bruteforce(True)
