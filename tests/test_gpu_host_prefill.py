"""GPU parity of gdn_prefill_host (host buffers, pieces of the sequence with
copies overlapping the prefills) against the fp64 oracle and against the
device-buffer prefill, through the C ABI.  Tolerance as for the bf16 prefill:
max|gpu - oracle| / max|oracle| <= 2e-2."""
import pytest
import torch

import oracle
from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn
from linear_attention_recurrence_14_b300.inputs import make_prefill_inputs

from .helpers import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _host(x):
    return {n: (None if getattr(x, n) is None else getattr(x, n).cpu().pin_memory())
            for n in ("q", "k", "v", "alpha", "beta", "S0")}


@pytest.mark.parametrize("B,T,Hqk,Hv,s0,tpp", [(2, 777, 2, 4, 0.02, 128), (1, 1000, 1, 2, 0.0, 0),
                                               (1, 300, 2, 2, 0.05, 1000), (2, 64, 1, 2, 0.02, 64),
                                               (1, 130, 1, 2, 0.02, 7)])
def test_host_prefill_matches_oracle(B, T, Hqk, Hv, s0, tpp):
    x = make_prefill_inputs(B, T, Hqk, Hv, 128, "bf16", decay_scale=0.1, s0_std=s0, seed=T + tpp, device="cpu")
    h = _host(x)
    shape = gdn.shape_of(x.q, x.v)
    ws = gdn.new_host_workspace(shape, "cuda", tpp)
    y, S_T = gdn.prefill_host(h["q"], h["k"], h["v"], h["alpha"], h["beta"], h["S0"], workspace=ws,
                              tokens_per_piece=tpp)
    torch.cuda.synchronize()
    assert gdn.read_device_status(ws) == 0
    yo, So = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    assert rel_err(y, yo) <= TOL[torch.bfloat16]
    assert rel_err(S_T, So) <= TOL[torch.bfloat16]


def test_host_prefill_agrees_with_device_prefill_and_empty():
    x = make_prefill_inputs(1, 2048, 2, 4, 128, "bf16", decay_scale=0.05, s0_std=0.02, seed=3, device="cpu")
    h = _host(x)
    y, S_T = gdn.prefill_host(h["q"], h["k"], h["v"], h["alpha"], h["beta"], h["S0"], tokens_per_piece=256)
    c = {n: h[n].cuda() for n in h}   # the same values on the device
    yd, Sd = gdn.prefill(c["q"], c["k"], c["v"], c["alpha"], c["beta"], c["S0"], segments=1)
    torch.cuda.synchronize()
    assert rel_err(y, yd.double().cpu().numpy()) <= 1e-2
    assert rel_err(S_T, Sd.double().cpu().numpy()) <= 1e-2
    e = make_prefill_inputs(1, 0, 1, 2, 128, "bf16", s0_std=0.05, seed=4, device="cpu")
    he = _host(e)
    ye, Se = gdn.prefill_host(he["q"], he["k"], he["v"], he["alpha"], he["beta"], he["S0"])
    torch.cuda.synchronize()
    assert ye.numel() == 0 and torch.equal(Se, e.S0)
