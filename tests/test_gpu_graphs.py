"""The library's calls captured into CUDA graphs and replayed: the chunked
prefill (four launches when the exact sequence split is taken), a run of
decode steps, and the chunked backward.  Each entry point does its host-side
setup (kernel attributes, device queries, tensor maps) on the first call, so a
call made before capture leaves only stream work to record.  Replays must
reproduce the eager results exactly (the same kernels on the same inputs)."""
import pytest
import torch

from linear_attention_recurrence_14_b300 import build as gbuild
from linear_attention_recurrence_14_b300 import gdn
from linear_attention_recurrence_14_b300.inputs import make_backward_grads, make_decode_inputs, make_prefill_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()


def test_prefill_with_exact_split_replays_from_a_graph():
    x = make_prefill_inputs(1, 64 * 300, 1, 2, 128, "bf16", decay_scale=0.0, s0_std=0.02, seed=101, device="cuda")
    shape = gdn.shape_of(x.q, x.v)
    assert gdn.prefill_launches(shape, segments=5) == 4
    ws = gdn.new_workspace(shape, "cuda")
    y, S_T = torch.empty_like(x.v), torch.empty_like(x.S0)
    run = lambda: gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, y=y, S_T=S_T, workspace=ws, segments=5)  # noqa: E731
    run()
    torch.cuda.synchronize()
    y_ref, S_ref = y.clone(), S_T.clone()
    y.zero_()
    S_T.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    g.replay()
    torch.cuda.synchronize()
    assert gdn.read_device_status(ws) == 0
    assert torch.equal(y, y_ref) and torch.equal(S_T, S_ref)


def test_decode_steps_replay_from_a_graph():
    steps = 16
    d = make_decode_inputs(8, steps, 2, 4, 128, "bf16", seed=102, device="cuda")
    ys = torch.empty((steps,) + tuple(d.v.shape[1:]), dtype=d.v.dtype, device="cuda")
    S = d.S0.clone()
    for s in range(steps):
        gdn.decode_step(d.q[s], d.k[s], d.v[s], d.alpha[s], d.beta[s], S, y=ys[s])
    torch.cuda.synchronize()
    y_ref, S_ref = ys.clone(), S.clone()
    S.copy_(d.S0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for s in range(steps):
            gdn.decode_step(d.q[s], d.k[s], d.v[s], d.alpha[s], d.beta[s], S, y=ys[s])
    S.copy_(d.S0)
    ys.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ys, y_ref) and torch.equal(S, S_ref)


def test_chunked_backward_replays_from_a_graph():
    x = make_prefill_inputs(1, 700, 1, 2, 128, "bf16", decay_scale=0.1, s0_std=0.02, seed=103, device="cuda")
    gr = make_backward_grads(1, 700, 2, 128, "bf16", ds_std=1.0, seed=103, device="cuda")
    shape = gdn.shape_of(x.q, x.v)
    ws = gdn.new_backward_workspace(shape, "cuda", chunked=True)
    out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, gr.dy, gr.dS_T, workspace=ws,
                       algorithm=gdn.ALGO_CHUNKED)
    torch.cuda.synchronize()
    ref = {n: t.clone() for n, t in out.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, gr.dy, gr.dS_T, out=out, workspace=ws,
                     algorithm=gdn.ALGO_CHUNKED)
    for t in out.values():
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for n in ref:
        assert torch.equal(out[n], ref[n]), n
