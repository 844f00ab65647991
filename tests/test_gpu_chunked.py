"""GPU parity of the chunked tensor-core prefill (bf16 q/k/v, fp32 gates and
state) against the fp64 oracle, through the C ABI.

Tolerance: max|gpu - oracle| / max|oracle| <= 2e-2 over each compared tensor
(bf16 inputs with an fp32 state)."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn
from linear_attention_recurrence_14_b300.inputs import make_prefill_inputs, workload_inputs

from .helpers import TOL, rel_err

pytestmark = pytest.mark.gpu
BF16_TOL = TOL[torch.bfloat16]


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _chunked(x, **kw):
    """Chunked prefill through the C ABI; also checks that no bounded device-side
    wait timed out (the kernel records that in the workspace status word)."""
    ws = gdn.new_workspace(gdn.shape_of(x.q, x.v), x.v.device)
    out = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, algorithm=gdn.ALGO_CHUNKED, workspace=ws, **kw)
    assert gdn.read_device_status(ws) == 0, "device-side wait timed out"
    return out


def test_chunked_repeated_launches_report_no_device_error():
    # Many launches of a multi-segment shape: a scheduling hazard in the
    # warp-specialised pipeline shows up as a timed-out bounded wait.
    x = make_prefill_inputs(1, 8192, 2, 4, 128, "bf16", decay_scale=0.05, s0_std=0.02, seed=21, device="cuda")
    ws = gdn.new_workspace(gdn.shape_of(x.q, x.v), "cuda")
    y = torch.empty_like(x.v)
    S = torch.empty_like(x.S0)
    for P in (1, 2, 3, 9, 16):
        for _ in range(20):
            gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, y=y, S_T=S, workspace=ws, algorithm=gdn.ALGO_CHUNKED,
                        segments=P)
        assert gdn.read_device_status(ws) == 0, f"device-side wait timed out with {P} segments"


@pytest.mark.parametrize(
    "B,T,Hqk,Hv,d,s0,segments,decay",
    [
        (1, 64, 1, 1, 128, 0.0, 1, 0.1),      # one full chunk
        (1, 1, 1, 1, 128, 0.02, 1, 0.1),      # a single token
        (1, 65, 1, 2, 128, 0.02, 1, 0.1),     # ragged tail
        (2, 200, 2, 4, 128, 0.02, 1, 0.1),    # grouped heads, several chunks
        (1, 300, 2, 2, 64, 0.05, 1, 0.1),     # d = 64 (zero-padded to the 128 tile)
        (2, 777, 1, 2, 128, 0.02, 3, 0.1),    # segments with warm-up windows
        (1, 1024, 2, 2, 128, 0.0, 7, 0.1),
        (1, 640, 1, 2, 128, 0.02, 2, 1.5),    # strong decay: every chunk below e^-40 (exact gate path)
        (1, 1280, 1, 2, 128, 0.02, 1, 0.6),   # chunks on both sides of the e^-40 switch
    ],
)
def test_chunked_small_matches_oracle(B, T, Hqk, Hv, d, s0, segments, decay):
    x = make_prefill_inputs(B, T, Hqk, Hv, d, "bf16", decay_scale=decay, s0_std=s0, seed=T + d, device="cuda")
    y, S_T = _chunked(x, segments=segments)
    yo, So = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    assert rel_err(y, yo) <= BF16_TOL
    assert rel_err(S_T, So) <= BF16_TOL


def test_chunked_train_workload_matches_oracle():
    # B=2, H=16, T=4096, d=128, S0 = 0: whole y and S_T, in the launch
    # configuration the library picks.
    x = workload_inputs("train", device="cuda")
    y, S_T = _chunked(x)
    yo, So = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    assert rel_err(y, yo) <= BF16_TOL
    assert rel_err(S_T, So) <= BF16_TOL


def test_chunked_grouped_workload_matches_oracle():
    # B=1, Hqk=16, Hv=32, T=65536, d=128, S0 ~ N(0, 0.02^2): whole y and S_T.
    x = workload_inputs("grouped", device="cuda")
    y, S_T = _chunked(x)
    yo, So = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    assert rel_err(y, yo) <= BF16_TOL
    assert rel_err(S_T, So) <= BF16_TOL


def _window_oracle(x, t0, t1, warm):
    """Oracle y over tokens [t0, t1) of every value head of batch 0 and the
    states at t1, started from a zero state `warm` tokens before t0 (from S0 at
    token 0 if the window reaches it).  With unit keys and beta in [0, 1] every
    step is a contraction of norm <= alpha_t, so the start-state difference is
    damped by the product of the gates over the warm-up, far below the
    tolerance for the warm-up lengths used here."""
    s = max(0, t0 - warm)
    sl = lambda t: t[0:1, s:t1]  # noqa: E731
    S0 = x.S0[0:1] if (s == 0 and x.S0 is not None) else None
    y, St = oracle.recurrence(sl(x.q), sl(x.k), sl(x.v), sl(x.alpha), sl(x.beta), S0)
    if t0 > s:
        damp = float(torch.exp(torch.log(x.alpha[0, s:t0].double()).sum(0)).max())
        assert damp < 1e-6, "warm-up too short for an exact window"
    return y[0, t0 - s:], St[0]


@pytest.mark.slow
def test_chunked_long_workload_windows_match_oracle():
    # B=1, H=16, T=2^20, d=128, gate scale 0.01: sampled windows of all sixteen
    # heads (start, across segment boundaries, end) and their final states.
    x = workload_inputs("long", device="cuda")
    T = x.q.shape[1]
    y, S_T = _chunked(x)
    errs = []
    for t0, t1 in ((0, 4096), (T // 2 - 3000, T // 2 + 3000), (T - 4096, T)):
        yo, So = _window_oracle(x, t0, t1, warm=8192)
        for hv in range(x.v.shape[2]):
            errs.append(rel_err(y[0, t0:t1, hv], yo[:, hv]))
            if t1 == T:
                errs.append(rel_err(S_T[0, hv], So[hv]))
    assert len(errs) == 3 * 16 + 16
    assert max(errs) <= BF16_TOL, errs


def test_chunked_segments_agree_with_single_pass():
    x = make_prefill_inputs(1, 4096, 2, 4, 128, "bf16", decay_scale=0.05, s0_std=0.02, seed=11, device="cuda")
    y1, S1 = _chunked(x, segments=1)
    for P in (2, 5, 16):
        yP, SP = _chunked(x, segments=P)
        assert rel_err(yP, y1.double().cpu().numpy()) <= 1e-2
        assert rel_err(SP, S1.double().cpu().numpy()) <= 1e-2


def test_chunked_in_place_state_and_empty():
    x = make_prefill_inputs(1, 500, 1, 2, 128, "bf16", decay_scale=0.1, s0_std=0.05, seed=12, device="cuda")
    yo, So = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    S = x.S0.clone()
    y, _ = _chunked(x, S_T=S, segments=3)
    assert rel_err(y, yo) <= BF16_TOL
    assert rel_err(S, So) <= BF16_TOL
    e = make_prefill_inputs(1, 0, 1, 2, 128, "bf16", s0_std=0.05, seed=13, device="cuda")
    y, S_T = _chunked(e)
    assert y.numel() == 0 and torch.equal(S_T, e.S0)


def test_chunked_identity_gates_keep_state():
    # alpha = 1, beta = 0: S_T = S0 and y_t = S0^T q_t (up to bf16 operand rounding).
    x = make_prefill_inputs(1, 256, 1, 2, 128, "bf16", s0_std=0.05, seed=14, device="cuda")
    x.alpha.fill_(1.0)
    x.beta.zero_()
    y, S_T = _chunked(x, segments=1)
    assert torch.equal(S_T, x.S0)
    yo, _ = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    assert rel_err(y, yo) <= BF16_TOL


def test_chunked_is_deterministic():
    x = make_prefill_inputs(1, 3000, 2, 4, 128, "bf16", s0_std=0.02, seed=15, device="cuda")
    y1, S1 = _chunked(x)
    y2, S2 = _chunked(x)
    assert torch.equal(y1, y2) and torch.equal(S1, S2)


def test_chunked_matches_sequential_kernel_and_decode():
    # Three independent paths of the library agree: chunked prefill,
    # token-sequential prefill, and T decode steps.
    x = make_prefill_inputs(2, 96, 1, 2, 128, "bf16", decay_scale=0.05, s0_std=0.02, seed=16, device="cuda")
    yc, Sc = _chunked(x)
    ys, Ss = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, algorithm=gdn.ALGO_SEQUENTIAL)
    S = x.S0.clone()
    tok = lambda a, t: a[:, t:t + 1].contiguous()  # noqa: E731
    yd = torch.stack([gdn.decode_step(tok(x.q, t), tok(x.k, t), tok(x.v, t), tok(x.alpha, t), tok(x.beta, t), S)
                      for t in range(96)], 1)[:, :, 0]
    ref = ys.double().cpu().numpy()
    assert rel_err(yc, ref) <= BF16_TOL
    assert rel_err(yd, ref) <= 1e-2
    assert rel_err(Sc, Ss.double().cpu().numpy()) <= BF16_TOL
    assert rel_err(S, Ss.double().cpu().numpy()) <= 1e-3


# ----------------------------------------------------------------------------
# Exact sequence split.  When a segment's preceding tokens do not forget the
# state within the warm-up limit (gates at or near 1), every segment is an
# affine map of its entering state (the reading notes' transition form,
# S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, composed over the
# segment): its two transition runs (from zero with the values, from the
# identity without them) and a short combine give each segment its exact start.
# The split is taken from 256 chunks of 64 tokens per sequence up; shorter
# sequences restart such segments from token 0.

def _oracle_check(x, y, S_T):
    yo, So = oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0)
    assert rel_err(y, yo) <= BF16_TOL
    assert rel_err(S_T, So) <= BF16_TOL


@pytest.mark.parametrize("segments", [3, 7])
@pytest.mark.parametrize("decay", [1.2e-4, 0.0])   # alpha ~ 1 - 1e-4, and alpha == 1 exactly
def test_exact_split_for_gates_that_do_not_decay(segments, decay):
    x = make_prefill_inputs(1, 64 * 256 + 5, 2, 4, 128, "bf16", decay_scale=decay, s0_std=0.02, seed=53, device="cuda")
    y, S_T = _chunked(x, segments=segments)
    _oracle_check(x, y, S_T)


def test_exact_split_mixed_heads_and_in_place_state():
    # Per head: strong decay (windows exist, no split) and no decay (split) in one call,
    # grouped value heads, a ragged tail, d = 64, and S_T written in place over S0.
    x = make_prefill_inputs(2, 64 * 256 + 17, 1, 4, 64, "bf16", decay_scale=0.05, s0_std=0.05, seed=59, device="cuda")
    x.alpha[:, :, 1] = 1.0
    x.alpha[:, :, 3] = 1.0 - 1e-5
    xr = make_prefill_inputs(2, 64 * 256 + 17, 1, 4, 64, "bf16", decay_scale=0.05, s0_std=0.05, seed=59, device="cuda")
    xr.alpha.copy_(x.alpha)
    S = x.S0.clone()
    ws = gdn.new_workspace(gdn.shape_of(x.q, x.v), "cuda")
    y, S_T = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, S, S_T=S, workspace=ws, algorithm=gdn.ALGO_CHUNKED,
                         segments=5)
    assert gdn.read_device_status(ws) == 0
    assert S_T.data_ptr() == S.data_ptr()
    _oracle_check(xr, y, S_T)


def test_exact_split_matches_the_single_pass():
    # The split must agree with one sequential pass of the same kernel (segments = 1)
    # far more closely than with the oracle: only the rounding order differs.
    x = make_prefill_inputs(1, 64 * 260, 1, 2, 128, "bf16", decay_scale=0.0, s0_std=0.02, seed=61, device="cuda")
    y1, S1 = _chunked(x, segments=1)
    y9, S9 = _chunked(x, segments=9)
    assert rel_err(y9, y1.double().cpu().numpy()) <= BF16_TOL
    assert rel_err(S9, S1.double().cpu().numpy()) <= BF16_TOL


def test_short_sequence_restarts_instead_of_splitting():
    # Below 256 chunks a segment without a window restarts from token 0: still exact.
    x = make_prefill_inputs(1, 64 * 40 + 5, 2, 4, 128, "bf16", decay_scale=0.0, s0_std=0.02, seed=67, device="cuda")
    y, S_T = _chunked(x, segments=5)
    _oracle_check(x, y, S_T)


def test_prefill_launch_counts():
    # gdn_prefill_launches: 4 kernels when the exact split is taken (long bf16 sequences over several
    # segments with a full workspace), else 1; 0 for an empty problem.
    big = gdn.GdnShape(1, 64 * 1024, 16, 32, 128, 128, gdn.GDN_BF16)   # the grouped shape
    assert gdn.prefill_launches(big) == 4
    assert gdn.prefill_launches(big, segments=1) == 1                  # one segment: nothing to split
    assert gdn.prefill_launches(big, algorithm=gdn.ALGO_SEQUENTIAL) == 1
    train = gdn.GdnShape(2, 4096, 16, 16, 128, 128, gdn.GDN_BF16)     # 64 chunks: restarts, no split
    assert gdn.prefill_launches(train) == 1
    assert gdn.prefill_launches(gdn.GdnShape(1, 0, 1, 2, 128, 128, gdn.GDN_BF16)) == 0
