"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

None of these re-types the oracle's loop: each checks it against a closed
form, an invariant, a brute-force evaluation of the equivalent transition
matrix (a different expression of the same map), or hand-worked numbers.
Citations: Qwen3.8-Next reading notes (jianyuh.github.io), section 2.1
"Gated DeltaNet" -- the four-line recurrence, the boxed transition-matrix form
S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, and the
erase-and-write paragraph.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, B, T, Hqk, Hv, dk, dv, unit_keys=True, alpha_range=(0.3, 1.0)):
    q = rng.standard_normal((B, T, Hqk, dk))
    k = rng.standard_normal((B, T, Hqk, dk))
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, dv))
    alpha = rng.uniform(*alpha_range, size=(B, T, Hv))
    beta = rng.uniform(0.0, 1.0, size=(B, T, Hv))
    S0 = rng.standard_normal((B, Hv, dk, dv))
    return q, k, v, alpha, beta, S0


def _transition_bruteforce(q, k, v, alpha, beta, S0):
    """Evaluate the boxed transition form as explicit matrix products.

    For each token t: S_t = (A_t ... A_1) S0 + sum_{tau<=t} (A_t ... A_{tau+1}) beta_tau k_tau v_tau^T
    with A_s = alpha_s (I - beta_s k_s k_s^T), every product formed explicitly.
    """
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    G = Hv // Hqk
    y = np.zeros((B, T, Hv, dv))
    S_T = np.zeros((B, Hv, dk, dv))
    I = np.eye(dk)
    for b in range(B):
        for h in range(Hv):
            hk = h // G
            A = [alpha[b, s, h] * (I - beta[b, s, h] * np.outer(k[b, s, hk], k[b, s, hk])) for s in range(T)]
            St = S0[b, h].copy() if T == 0 else None
            for t in range(T):
                prod = np.eye(dk)
                for s in range(t, -1, -1):
                    prod = prod @ A[s]
                St = prod @ S0[b, h]
                for tau in range(t + 1):
                    P = np.eye(dk)
                    for s in range(t, tau, -1):
                        P = P @ A[s]
                    St = St + P @ (beta[b, tau, h] * np.outer(k[b, tau, hk], v[b, tau, h]))
                y[b, t, h] = St.T @ q[b, t, hk]
            S_T[b, h] = St
    return y, S_T


@pytest.mark.parametrize("unit_keys", [True, False])
def test_transition_matrix_bruteforce(unit_keys):
    # dk != dv and G = 2 with distinct key heads: a transposed operand, a wrong
    # head mapping or a dropped term all change the result.
    rng = np.random.default_rng(1)
    q, k, v, alpha, beta, S0 = _rand_inputs(rng, 2, 9, 2, 4, 5, 3, unit_keys=unit_keys)
    y, S_T = oracle.recurrence(q, k, v, alpha, beta, S0)
    yb, Sb = _transition_bruteforce(q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(y, yb, rtol=0, atol=1e-12 * max(1.0, np.abs(yb).max()))
    np.testing.assert_allclose(S_T, Sb, rtol=0, atol=1e-12 * max(1.0, np.abs(Sb).max()))


def test_transition_bruteforce_t16():
    rng = np.random.default_rng(2)
    q, k, v, alpha, beta, S0 = _rand_inputs(rng, 1, 16, 1, 1, 6, 6)
    y, S_T = oracle.recurrence(q, k, v, alpha, beta, S0)
    yb, Sb = _transition_bruteforce(q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(y, yb, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S_T, Sb, rtol=0, atol=1e-12)


def test_identity_gates_keep_state():
    # alpha = 1, beta = 0: nothing decays, nothing is written, y_t = S0^T q_t.
    rng = np.random.default_rng(3)
    q, k, v, alpha, beta, S0 = _rand_inputs(rng, 2, 7, 1, 2, 4, 6)
    alpha[:] = 1.0
    beta[:] = 0.0
    y, S_T = oracle.recurrence(q, k, v, alpha, beta, S0)
    np.testing.assert_array_equal(S_T, S0)
    expect = np.einsum("bhij,bti->bthj", S0, q[:, :, 0, :])
    np.testing.assert_allclose(y, expect, rtol=0, atol=1e-13)


def test_beta_zero_is_pure_decay():
    # beta = 0: S_t = (prod_{s<=t} alpha_s) S0 and y_t = S_t^T q_t.
    rng = np.random.default_rng(4)
    q, k, v, alpha, beta, S0 = _rand_inputs(rng, 1, 11, 1, 1, 4, 4)
    beta[:] = 0.0
    y, S_T = oracle.recurrence(q, k, v, alpha, beta, S0)
    cum = np.cumprod(alpha[0, :, 0])
    np.testing.assert_allclose(S_T[0, 0], cum[-1] * S0[0, 0], rtol=1e-14, atol=0)
    expect = cum[:, None] * (q[0, :, 0, :] @ S0[0, 0])
    np.testing.assert_allclose(y[0, :, 0], expect, rtol=1e-13, atol=1e-15)


def test_orthonormal_keys_store_and_retrieve():
    # alpha = beta = 1, S0 = 0, orthonormal keys: every written value is stored
    # exactly and a later read with beta = 0 and q = k_j returns v_j.
    rng = np.random.default_rng(5)
    dk, dv, n = 8, 5, 8
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm.T[:n]                      # rows are orthonormal
    vals = rng.standard_normal((n, dv))
    order = rng.permutation(n)
    T = 2 * n
    k = np.zeros((1, T, 1, dk))
    q = np.zeros((1, T, 1, dk))
    v = np.zeros((1, T, 1, dv))
    beta = np.zeros((1, T, 1))
    alpha = np.ones((1, T, 1))
    k[0, :n, 0] = keys
    q[0, :n, 0] = keys
    v[0, :n, 0] = vals
    beta[0, :n, 0] = 1.0
    q[0, n:, 0] = keys[order]            # reads, nothing written (beta = 0)
    k[0, n:, 0] = keys[order]
    y, S_T = oracle.recurrence(q, k, v, alpha, beta, None)
    np.testing.assert_allclose(y[0, :n, 0], vals, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[0, n:, 0], vals[order], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S_T[0, 0], keys.T @ vals, rtol=0, atol=1e-12)


def test_repeated_key_overwrites():
    # The delta rule erases before it writes: the same unit key written twice
    # with alpha = beta = 1 leaves S = k v2^T, not k (v1 + v2)^T.
    rng = np.random.default_rng(6)
    dk, dv = 6, 4
    kk = rng.standard_normal(dk)
    kk /= np.linalg.norm(kk)
    v1, v2 = rng.standard_normal(dv), rng.standard_normal(dv)
    k = np.stack([kk, kk])[None, :, None, :]
    q = k.copy()
    v = np.stack([v1, v2])[None, :, None, :]
    ones = np.ones((1, 2, 1))
    y, S_T = oracle.recurrence(q, k, v, ones, ones, None)
    np.testing.assert_allclose(S_T[0, 0], np.outer(kk, v2), rtol=0, atol=1e-14)
    np.testing.assert_allclose(y[0, 1, 0], v2, rtol=0, atol=1e-14)


def test_single_step_from_zero_state():
    # From S0 = 0 one step gives y_1 = beta_1 (k_1 . q_1) v_1, whatever alpha_1 is:
    # the output is read after the write.
    rng = np.random.default_rng(7)
    for a in (0.1, 0.5, 1.0):
        q, k, v, alpha, beta, _ = _rand_inputs(rng, 1, 1, 1, 1, 5, 3)
        alpha[:] = a
        y, _ = oracle.recurrence(q, k, v, alpha, beta, None)
        expect = beta[0, 0, 0] * (k[0, 0, 0] @ q[0, 0, 0]) * v[0, 0, 0]
        np.testing.assert_allclose(y[0, 0, 0], expect, rtol=1e-14, atol=1e-16)


def test_decay_applies_before_the_residual():
    # One step from a random state with alpha < 1 follows the equations
    # (e formed from the decayed state), not the walkthrough snippet that forms
    # e from the undecayed state.
    rng = np.random.default_rng(8)
    q, k, v, alpha, beta, S0 = _rand_inputs(rng, 1, 1, 1, 1, 4, 4)
    alpha[:] = 0.6
    y, S_T = oracle.recurrence(q, k, v, alpha, beta, S0)
    kk, vv, a, b = k[0, 0, 0], v[0, 0, 0], 0.6, beta[0, 0, 0]
    boxed = a * (np.eye(4) - b * np.outer(kk, kk)) @ S0[0, 0] + b * np.outer(kk, vv)
    variant = (a * np.eye(4) - b * np.outer(kk, kk)) @ S0[0, 0] + b * np.outer(kk, vv)
    np.testing.assert_allclose(S_T[0, 0], boxed, rtol=0, atol=1e-14)
    assert np.abs(S_T[0, 0] - variant).max() > 1e-3


def test_contraction_bound():
    # With unit keys and beta in [0, 1] the homogeneous map is a contraction:
    # ||alpha (I - beta k k^T)||_2 <= alpha, so two runs that differ only in S0
    # differ at the end by at most prod(alpha) * ||dS0||_2 (spectral norm).
    rng = np.random.default_rng(9)
    q, k, v, alpha, beta, S0 = _rand_inputs(rng, 1, 40, 1, 1, 6, 5, alpha_range=(0.8, 1.0))
    S0b = S0 + rng.standard_normal(S0.shape)
    _, Sa = oracle.recurrence(q, k, v, alpha, beta, S0)
    _, Sb = oracle.recurrence(q, k, v, alpha, beta, S0b)
    lhs = np.linalg.norm(Sa[0, 0] - Sb[0, 0], 2)
    rhs = np.prod(alpha[0, :, 0]) * np.linalg.norm(S0[0, 0] - S0b[0, 0], 2)
    assert lhs <= rhs * (1 + 1e-12)


def test_empty_sequence_returns_initial_state():
    rng = np.random.default_rng(10)
    q, k, v, alpha, beta, S0 = _rand_inputs(rng, 2, 0, 1, 2, 4, 4)
    y, S_T = oracle.recurrence(q, k, v, alpha, beta, S0)
    assert y.shape == (2, 0, 2, 4)
    np.testing.assert_array_equal(S_T, S0)


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out[key] = np.array([float(x) for x in val.split()])
    return out


def test_golden_hand_worked_example():
    g = _read_golden("hand_worked_d2.txt")
    dk, dv = int(g["dk"][0]), int(g["dv"][0])
    T = len(g["alpha"])
    y, S_T = oracle.recurrence(
        g["q"].reshape(1, T, 1, dk), g["k"].reshape(1, T, 1, dk), g["v"].reshape(1, T, 1, dv),
        g["alpha"].reshape(1, T, 1), g["beta"].reshape(1, T, 1), g["S0"].reshape(1, 1, dk, dv))
    np.testing.assert_allclose(y.ravel(), g["y"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S_T.ravel(), g["S_T"], rtol=0, atol=1e-12)


def test_head_slice_matches_full_run():
    # The per-pair helper used by the large parity tests slices the right key head.
    rng = np.random.default_rng(11)
    q, k, v, alpha, beta, S0 = _rand_inputs(rng, 2, 5, 2, 4, 3, 3)
    y, S_T = oracle.recurrence(q, k, v, alpha, beta, S0)
    for b, h in [(0, 0), (1, 3), (0, 2)]:
        yh, sh = oracle.recurrence_head(q, k, v, alpha, beta, S0, b, h)
        np.testing.assert_array_equal(yh, y[b, :, h])
        np.testing.assert_array_equal(sh, S_T[b, h])
