"""The method's degenerate cases on the GPU, through the C ABI, for every path
that runs the recurrence: the chunked tensor-core prefill (bf16), the
token-sequential prefill (bf16 and fp32) and the decode step (bf16 and fp32).

Each case has a closed form from the recurrence of the reading notes, section
2.1 "Gated DeltaNet" (S~ = alpha S, e = v - S~^T k, S = S~ + beta k e^T,
y = S^T q), and the kernels are compared with both that closed form and the
fp64 oracle.  Keys are built to be exactly orthonormal in bf16: rows of a
64 x 64 Hadamard matrix scaled by 1/8 (entries +-1/8, unit norm), placed on
one of two disjoint 64-coordinate halves of a d = 128 key and then permuted
and sign-flipped per coordinate, so 128 mutually orthogonal unit keys exist
and every inner product of two of them is exact in any precision."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn

from .helpers import TOL, rel_err

pytestmark = pytest.mark.gpu
D = 128

# (name, dtype, prefill algorithm or None for the decode step)
PATHS = [("chunked", torch.bfloat16, gdn.ALGO_CHUNKED), ("sequential-bf16", torch.bfloat16, gdn.ALGO_SEQUENTIAL),
         ("sequential-f32", torch.float32, gdn.ALGO_SEQUENTIAL), ("decode-bf16", torch.bfloat16, None),
         ("decode-f32", torch.float32, None)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _hadamard(n):
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def _orthonormal_keys(seed):
    """128 x 128 matrix whose rows are orthonormal unit keys with entries in {0, +-1/8}."""
    rng = np.random.default_rng(seed)
    h = _hadamard(64) / 8.0
    keys = np.zeros((D, D))
    keys[:64, :64] = h
    keys[64:, 64:] = h
    keys = keys[:, rng.permutation(D)] * rng.choice([-1.0, 1.0], size=D)[None, :]
    return keys[rng.permutation(D)]


def _run(path, q, k, v, alpha, beta, S0):
    """Run one path on fp64 host arrays [T, d] (one batch, one head); returns y [T, dv], S_T [dk, dv]."""
    name, dt, algo = path
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dt)  # noqa: E731
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.float32)  # noqa: E731
    T = q.shape[0]
    if algo is not None:
        ws = gdn.new_workspace(gdn.shape_of(to(q[None, :, None]), to(v[None, :, None])), "cuda")
        y, S_T = gdn.prefill(to(q[None, :, None]), to(k[None, :, None]), to(v[None, :, None]),
                             g(alpha[None, :, None]), g(beta[None, :, None]),
                             None if S0 is None else g(S0[None, None]), workspace=ws, algorithm=algo)
        assert gdn.read_device_status(ws) == 0
        torch.cuda.synchronize()
        return y[0, :, 0].double().cpu().numpy(), S_T[0, 0].double().cpu().numpy()
    S = g(np.zeros((1, 1, D, D)) if S0 is None else S0[None, None])
    ys = []
    for t in range(T):
        ys.append(gdn.decode_step(to(q[None, t:t + 1, None]), to(k[None, t:t + 1, None]), to(v[None, t:t + 1, None]),
                                  g(alpha[None, t:t + 1, None]), g(beta[None, t:t + 1, None]), S)[0, 0, 0])
    torch.cuda.synchronize()
    return torch.stack(ys).double().cpu().numpy(), S[0, 0].double().cpu().numpy()


def _oracle(q, k, v, alpha, beta, S0):
    y, S_T = oracle.recurrence(q[None, :, None], k[None, :, None], v[None, :, None], alpha[None, :, None],
                               beta[None, :, None], None if S0 is None else S0[None, None])
    return y[0, :, 0], S_T[0, 0]


def _bf16(a):
    return torch.from_numpy(a).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_orthonormal_keys_store_and_retrieve(path):
    # alpha = beta = 1 from S0 = 0: 100 writes of orthonormal keys (across a chunk
    # boundary), then 100 reads in another order with beta = 0.  Each write reads
    # back its own value, each later read returns the value stored under its key,
    # and S_T = sum_j k_j v_j^T.
    rng = np.random.default_rng(71)
    n, T = 100, 200
    keys = _orthonormal_keys(72)[:n]
    vals = _bf16(rng.standard_normal((n, D)))
    order = rng.permutation(n)
    k = np.concatenate([keys, keys[order]])
    v = np.concatenate([vals, np.zeros((n, D))])
    beta = np.concatenate([np.ones(n), np.zeros(n)])
    alpha = np.ones(T)
    y, S_T = _run(path, k, k, v, alpha, beta, None)
    tol = TOL[path[1]]
    assert rel_err(y[:n], vals) <= tol
    assert rel_err(y[n:], vals[order]) <= tol
    assert rel_err(S_T, keys.T @ vals) <= tol
    yo, So = _oracle(k, k, v, alpha, beta, None)
    assert rel_err(y, yo) <= tol and rel_err(S_T, So) <= tol


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_repeated_key_overwrites(path):
    # The same unit key written at every one of 130 steps with alpha = beta = 1:
    # the delta rule erases before it writes, so each read (q = k) returns the
    # latest value and S_T = k v_T^T, not k (sum_t v_t)^T.  In the chunked form
    # every entry of the strictly lower A is 1 here, the hardest case of its
    # triangular solve.
    rng = np.random.default_rng(73)
    T = 130
    kk = _orthonormal_keys(74)[0]
    k = np.tile(kk, (T, 1))
    v = _bf16(rng.standard_normal((T, D)))
    ones = np.ones(T)
    y, S_T = _run(path, k, k, v, ones, ones, None)
    tol = TOL[path[1]]
    assert rel_err(y, v) <= tol
    assert rel_err(S_T, np.outer(kk, v[-1])) <= tol
    yo, So = _oracle(k, k, v, ones, ones, None)
    assert rel_err(y, yo) <= tol and rel_err(S_T, So) <= tol


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_one_step_decays_before_the_residual(path):
    # One step from a random state with alpha = 0.6:
    # S_1 = alpha (I - beta k k^T) S0 + beta k v^T, y_1 = S_1^T q.  The variant that
    # forms the residual from the undecayed state differs from it by far more
    # than the tolerance (the key is a coordinate vector, so the difference,
    # (alpha - 1) beta k k^T S0, is a whole row of S0).
    rng = np.random.default_rng(75)
    kk = np.zeros(D)
    kk[37] = 1.0
    q = rng.standard_normal(D)
    q = _bf16(q / np.linalg.norm(q))
    v = _bf16(0.1 * rng.standard_normal(D))
    S0 = rng.standard_normal((D, D))
    a, b = 0.6, 0.75
    y, S_T = _run(path, q[None], kk[None], v[None], np.array([a]), np.array([b]), S0)
    boxed = a * (np.eye(D) - b * np.outer(kk, kk)) @ S0 + b * np.outer(kk, v)
    variant = (a * np.eye(D) - b * np.outer(kk, kk)) @ S0 + b * np.outer(kk, v)
    tol = TOL[path[1]]
    assert rel_err(S_T, boxed) <= tol
    assert rel_err(y[0], boxed.T @ q) <= tol
    assert rel_err(variant, boxed) > 5 * TOL[torch.bfloat16]
