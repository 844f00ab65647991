"""GPU parity of the channel-wise decay entry points (gdn_prefill_cw,
gdn_decode_step_cw: S~ = diag(alpha_t) S) against the fp64 oracle's
channel-wise mode, through the C ABI.  Tolerances as for the scalar gate:
1e-4 (fp32 inputs) and 2e-2 (bf16 inputs), max|gpu - oracle| / max|oracle|."""
import ctypes

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


@pytest.mark.parametrize("algorithm,tol_y,tol_s", [(gdn.ALGO_SEQUENTIAL, 1e-2, 1e-3),
                                                   (gdn.ALGO_CHUNKED, TOL[torch.bfloat16], TOL[torch.bfloat16])])
def test_prefill_cw_in_place_and_uniform_channels_match_scalar(algorithm, tol_y, tol_s):
    # All channels equal: the scalar recurrence.  The token-sequential kernels (fp32
    # arithmetic on both sides) agree closely; the chunked path to the bf16 tolerance.
    x = make_prefill_inputs(1, 300, 2, 4, 128, "bf16", s0_std=0.02, seed=9, device="cuda")
    a_uniform = x.alpha[..., None].expand(-1, -1, -1, 128).contiguous()
    S = x.S0.clone()
    y, _ = gdn.prefill_cw(x.q, x.k, x.v, a_uniform, x.beta, S, S_T=S, algorithm=algorithm)
    ys, Ss = gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, algorithm=gdn.ALGO_SEQUENTIAL)
    assert rel_err(y, ys.double().cpu().numpy()) <= tol_y
    assert rel_err(S, Ss.double().cpu().numpy()) <= tol_s


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


# ----------------------------------------------------------------------------
# The chunked tensor-core path (bf16, d = 128): per-chunk pre-pass + chain kernel.

def _cw_chunked(x, a, **kw):
    return gdn.prefill_cw(x.q, x.k, x.v, a, x.beta, x.S0, algorithm=gdn.ALGO_CHUNKED, **kw)


@pytest.mark.parametrize("B,T,Hqk,Hv,s0,segments,decay", [
    (1, 64, 1, 1, 0.0, 1, 0.1),       # one whole chunk
    (1, 1, 1, 1, 0.02, 1, 0.1),       # a single token
    (1, 65, 1, 2, 0.02, 1, 0.1),      # ragged tail, grouped heads
    (2, 300, 2, 4, 0.02, 1, 0.05),    # several chunks
    (2, 777, 1, 2, 0.02, 3, 0.1),     # segments with warm-up windows
    (1, 1500, 2, 2, 0.05, 7, 0.5),    # strong decay: short windows
    (1, 640, 1, 2, 0.02, 4, 0.0),     # alpha = 1: no window, segments restart from token 0
    (1, 500, 1, 4, 0.02, 2, 0.1),     # four value heads per key head
])
def test_prefill_cw_chunked_matches_oracle(B, T, Hqk, Hv, s0, segments, decay):
    x = make_prefill_inputs(B, T, Hqk, Hv, 128, "bf16", s0_std=s0, seed=T + 7, device="cuda")
    a = make_channelwise_alpha(B, T, Hv, 128, decay_scale=decay, seed=T + 1, device="cuda")
    if decay == 0.0:
        a.fill_(1.0)
    y, S_T = _cw_chunked(x, a, segments=segments)
    yo, So = oracle.recurrence(x.q, x.k, x.v, a, x.beta, x.S0)
    assert rel_err(y, yo) <= TOL[torch.bfloat16]
    assert rel_err(S_T, So) <= TOL[torch.bfloat16]


def test_prefill_cw_chunked_channels_that_forget_at_once():
    # A quarter of the channels decay by alpha = 1e-3 per token (a 16-token block
    # decays by e^-110 there): those blocks take the element-wise path, the rest
    # of the chunk the scaled products.  Another quarter keeps alpha = 1.
    x = make_prefill_inputs(1, 200, 1, 2, 128, "bf16", s0_std=0.05, seed=81, device="cuda")
    a = make_channelwise_alpha(1, 200, 2, 128, decay_scale=0.1, seed=82, device="cuda")
    a[..., 0:32] = 1e-3
    a[..., 32:64] = 1.0
    a[:, 100:140, 1, 64:] = 1e-3    # and whole blocks of one head in every channel
    y, S_T = _cw_chunked(x, a, segments=2)
    yo, So = oracle.recurrence(x.q, x.k, x.v, a, x.beta, x.S0)
    assert rel_err(y, yo) <= TOL[torch.bfloat16]
    assert rel_err(S_T, So) <= TOL[torch.bfloat16]


def test_prefill_cw_chunked_in_place_and_agrees_with_sequential():
    x = make_prefill_inputs(2, 1000, 2, 4, 128, "bf16", s0_std=0.02, seed=83, device="cuda")
    a = make_channelwise_alpha(2, 1000, 4, 128, decay_scale=0.05, seed=84, device="cuda")
    ys, Ss = gdn.prefill_cw(x.q, x.k, x.v, a, x.beta, x.S0, algorithm=gdn.ALGO_SEQUENTIAL)
    S = x.S0.clone()
    y, _ = gdn.prefill_cw(x.q, x.k, x.v, a, x.beta, S, S_T=S, segments=5)   # auto: chunked
    assert rel_err(y, ys.double().cpu().numpy()) <= TOL[torch.bfloat16]
    assert rel_err(S, Ss.double().cpu().numpy()) <= TOL[torch.bfloat16]
    # the entry point without a workspace allocates its own and takes the same path
    y2, S2 = torch.empty_like(y), torch.empty_like(S)
    shape = gdn.shape_of(x.q, x.v)
    rc = gdn.lib().gdn_prefill_cw(ctypes.byref(shape), *(ctypes.c_void_p(t.data_ptr()) for t in
                                  (x.q, x.k, x.v, a, x.beta, x.S0, y2, S2)),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == gdn.GDN_OK
    torch.cuda.synchronize()
    yc, Sc = gdn.prefill_cw(x.q, x.k, x.v, a, x.beta, x.S0)
    assert torch.equal(y2, yc) and torch.equal(S2, Sc)


@pytest.mark.slow
def test_prefill_cw_chunked_grouped_shape_windows_match_oracle():
    # B=1, T=65536, 16 q/k heads, 32 v heads, d=128, per-channel gate scale 0.05:
    # windows (start, across segment boundaries, end) of four heads and their final states.
    x = make_prefill_inputs(1, 65536, 16, 32, 128, "bf16", s0_std=0.02, seed=85, device="cuda")
    a = make_channelwise_alpha(1, 65536, 32, 128, decay_scale=0.05, seed=86, device="cuda")
    y, S_T = gdn.prefill_cw(x.q, x.k, x.v, a, x.beta, x.S0)
    T = 65536
    errs = []
    for t0, t1 in ((0, 2048), (T // 2 - 1500, T // 2 + 1500), (T - 2048, T)):
        s = max(0, t0 - 6144)
        heads = [0, 11, 20, 31]
        hk = [h // 2 for h in heads]
        sl = lambda t, hh: t[:, s:t1, hh].contiguous()  # noqa: E731
        S0 = x.S0[:, heads] if s == 0 else None
        yo, So = oracle.recurrence(sl(x.q, hk), sl(x.k, hk), sl(x.v, heads), sl(a, heads), sl(x.beta, heads), S0)
        if s > 0:   # the window start is forgotten: max-channel decay over the warm-up below 1e-6
            damp = torch.exp(torch.log(a[0, s:t0, heads].double()).max(-1).values.sum(0)).max()
            assert float(damp) < 1e-6
        for i, h in enumerate(heads):
            errs.append(rel_err(y[0, t0:t1, h], yo[0, t0 - s:, i]))
            if t1 == T:
                errs.append(rel_err(S_T[0, h], So[0, i]))
    assert max(errs) <= TOL[torch.bfloat16], errs


def test_prefill_cw_chunked_exact_split_for_channels_that_do_not_decay():
    # A quarter of the channels keep alpha = 1, so no window of preceding chunks forgets the
    # state: over 256 chunks the chain takes the exact split (segment maps and their combine).
    T = 64 * 260 + 7
    x = make_prefill_inputs(1, T, 1, 2, 128, "bf16", s0_std=0.02, seed=95, device="cuda")
    a = make_channelwise_alpha(1, T, 2, 128, decay_scale=0.05, seed=96, device="cuda")
    a[..., 96:] = 1.0
    y, S_T = gdn.prefill_cw(x.q, x.k, x.v, a, x.beta, x.S0, segments=9)
    yo, So = oracle.recurrence(x.q, x.k, x.v, a, x.beta, x.S0)
    assert rel_err(y, yo) <= TOL[torch.bfloat16]
    assert rel_err(S_T, So) <= TOL[torch.bfloat16]
    # against one sequential pass of the same chain (segments = 1): only rounding order differs
    y1, S1 = gdn.prefill_cw(x.q, x.k, x.v, a, x.beta, x.S0, segments=1)
    assert rel_err(y, y1.double().cpu().numpy()) <= TOL[torch.bfloat16]
    assert rel_err(S_T, S1.double().cpu().numpy()) <= TOL[torch.bfloat16]


def test_prefill_cw_chunk_decay_bounds():
    # The pre-pass writes, per (batch, value head, chunk), the bound sum_t max_c log alpha_tc
    # (natural log) that the warm-up windows and the exact split's plan compare with
    # log_eps: the state's decay over the chunk is at most its exponential, since
    # ||diag(alpha)(I - beta k k^T)|| <= max_c alpha_c for unit keys and beta in [0, 1].
    # White-box: the bounds are the last B * Hv * nchunks floats of the chunked path's
    # workspace.  Checked against a host computation from the same alpha on a ragged
    # length with some channels at alpha = 1 and some strongly decaying.
    B, T, Hqk, Hv, d = 2, 1000, 1, 2, 128
    x = make_prefill_inputs(B, T, Hqk, Hv, d, "bf16", s0_std=0.02, seed=41, device="cuda")
    a = make_channelwise_alpha(B, T, Hv, d, decay_scale=0.3, seed=41, device="cuda")
    a[:, :, 0, :8] = 1.0
    a[:, 500:, 1, 100:] = 1e-3
    ws = gdn.new_cw_workspace(gdn.shape_of(x.q, x.v), "cuda")
    _cw_chunked(x, a, workspace=ws)
    torch.cuda.synchronize()
    nchunks = (T + 63) // 64
    n = B * Hv * nchunks
    got = ws[ws.numel() - 4 * n:].view(torch.float32).reshape(B, Hv, nchunks).double().cpu()
    la = torch.log(a.double().cpu()).amax(dim=3)                     # [B, T, Hv]
    la = torch.cat([la, torch.zeros(B, nchunks * 64 - T, Hv, dtype=la.dtype)], 1)
    want = la.reshape(B, nchunks, 64, Hv).sum(2).permute(0, 2, 1)   # [B, Hv, nchunks]
    # base-2 cumulative sums in fp32 with an approximate log2 (about 2^-22 per token)
    assert torch.allclose(got, want, rtol=1e-4, atol=2e-3), (got - want).abs().max()
    assert (got[:, 0, :] > -1e-4).all()   # the head with channels at alpha = 1 never decays
