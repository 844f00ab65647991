"""GPU parity of the token-sequential kernel (decode and the fp32 prefill path)
against the fp64 oracle, through the C ABI."""
import pytest
import torch

import oracle
from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn
from linear_attention_recurrence_14_b300.inputs import make_decode_inputs, make_prefill_inputs, workload_inputs

from .helpers import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def test_tiny_fp32_workload_matches_oracle():
    # B=1, H=2, T=256, d=64, fp32, S0 = 0: the whole output and final state.
    x = workload_inputs("tiny", device="cuda")
    y, S_T = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    yo, So = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    assert rel_err(y, yo) <= TOL[torch.float32]
    assert rel_err(S_T, So) <= TOL[torch.float32]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2])
def test_sequential_prefill_matches_oracle(dtype, d, G):
    x = make_prefill_inputs(2, 77, 2, 2 * G, d, dtype, decay_scale=0.1, s0_std=0.05, seed=3, device="cuda")
    y, S_T = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, algorithm=gdn.ALGO_SEQUENTIAL)
    yo, So = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    tol = TOL[x.q.dtype]
    assert rel_err(y, yo) <= tol
    assert rel_err(S_T, So) <= tol


def test_sequential_prefill_in_place_and_empty():
    x = make_prefill_inputs(1, 40, 1, 2, 64, "f32", decay_scale=0.1, s0_std=0.05, seed=4, device="cuda")
    So_ref = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)[1]
    S = x.S0.clone()
    gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, S, S_T=S)
    assert rel_err(S, So_ref) <= 1e-4
    e = make_prefill_inputs(1, 0, 1, 2, 64, "f32", s0_std=0.05, seed=5, device="cuda")
    y, S_T = gdn.prefill(e.q, e.k, e.v, e.alpha, e.beta, e.S0)
    assert y.numel() == 0
    assert torch.equal(S_T, e.S0)
    y, S_T = gdn.prefill(e.q, e.k, e.v, e.alpha, e.beta, None)
    assert torch.count_nonzero(S_T) == 0


def _decode_vs_oracle(x, steps):
    B = x.S0.shape[0]
    S = x.S0.clone()
    ys = []
    for s in range(steps):
        ys.append(gdn.decode_step(x.q[s], x.k[s], x.v[s], x.alpha[s], x.beta[s], S))
    y = torch.stack(ys, 0)  # [steps, B, 1, Hv, d]
    seq = lambda t: t[:, :, 0].transpose(0, 1).contiguous()  # noqa: E731  [B, steps, H, ...]
    yo, So = oracle.recurrence(seq(x.q), seq(x.k), seq(x.v), seq(x.alpha), seq(x.beta), x.S0)
    return rel_err(seq(y), yo), rel_err(S, So)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 128), ("bf16", 64), ("f32", 64)])
def test_decode_small_matches_oracle(dtype, d):
    x = make_decode_inputs(3, 6, 2, 4, d, dtype, decay_scale=0.05, s0_std=0.02, seed=6, device="cuda")
    ey, es = _decode_vs_oracle(x, 6)
    tol = TOL[x.q.dtype]
    assert ey <= tol and es <= tol


def test_decode_workload_matches_oracle():
    # B=256, Hv=32 over Hqk=16, d=128, 128 steps, state updated in place:
    # every step's y and the final state are compared.
    x = workload_inputs("decode", device="cuda")
    ey, es = _decode_vs_oracle(x, x.q.shape[0])
    assert ey <= TOL[torch.bfloat16]
    assert es <= TOL[torch.bfloat16]
