"""GPU parity of the channel-wise decay entry points (gdn_prefill_cw,
gdn_decode_step_cw: S~ = diag(alpha_t) S) against the fp64 oracle's
channel-wise mode, through the C ABI.  Tolerances as for the scalar gate:
1e-4 (fp32 inputs) and 2e-2 (bf16 inputs), max|gpu - oracle| / max|oracle|."""
import pytest
import torch

import oracle
from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn
from linear_attention_recurrence_14_b300.inputs import make_channelwise_alpha, make_prefill_inputs

from .helpers import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


@pytest.mark.parametrize("B,T,Hqk,Hv,d,dtype,s0", [(1, 200, 1, 2, 128, "bf16", 0.02), (2, 97, 2, 4, 128, "bf16", 0.0),
                                                  (1, 150, 2, 2, 64, "f32", 0.05), (1, 1, 1, 2, 128, "f32", 0.05),
                                                  (1, 0, 1, 2, 64, "f32", 0.05)])
def test_prefill_cw_matches_oracle(B, T, Hqk, Hv, d, dtype, s0):
    x = make_prefill_inputs(B, T, Hqk, Hv, d, dtype, s0_std=s0, seed=T + d, device="cuda")
    a = make_channelwise_alpha(B, T, Hv, d, decay_scale=0.1, seed=T, device="cuda")
    y, S_T = gdn.prefill_cw(x.q, x.k, x.v, a, x.beta, x.S0)
    yo, So = oracle.recurrence(x.q, x.k, x.v, a, x.beta, x.S0)
    tol = TOL[x.q.dtype]
    assert rel_err(y, yo) <= tol
    assert rel_err(S_T, So) <= tol


def test_prefill_cw_in_place_and_uniform_channels_match_scalar():
    x = make_prefill_inputs(1, 300, 2, 4, 128, "bf16", s0_std=0.02, seed=9, device="cuda")
    a_uniform = x.alpha[..., None].expand(-1, -1, -1, 128).contiguous()
    S = x.S0.clone()
    y, _ = gdn.prefill_cw(x.q, x.k, x.v, a_uniform, x.beta, S, S_T=S)
    ys, Ss = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, algorithm=gdn.ALGO_SEQUENTIAL)
    assert rel_err(y, ys.double().cpu().numpy()) <= 1e-2
    assert rel_err(S, Ss.double().cpu().numpy()) <= 1e-3


def test_decode_cw_steps_match_oracle():
    B, Hqk, Hv, d, steps = 8, 2, 4, 128, 6
    x = make_prefill_inputs(B, steps, Hqk, Hv, d, "bf16", s0_std=0.02, seed=11, device="cuda")
    a = make_channelwise_alpha(B, steps, Hv, d, decay_scale=0.05, seed=11, device="cuda")
    S = x.S0.clone()
    tok = lambda t_, i: t_[:, i:i + 1].contiguous()  # noqa: E731
    ys = [gdn.decode_step_cw(tok(x.q, i), tok(x.k, i), tok(x.v, i), tok(a, i), tok(x.beta, i), S)
          for i in range(steps)]
    yo, So = oracle.recurrence(x.q, x.k, x.v, a, x.beta, x.S0)
    assert rel_err(torch.cat(ys, 1), yo) <= TOL[torch.bfloat16]
    assert rel_err(S, So) <= TOL[torch.bfloat16]
