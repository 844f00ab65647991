"""Seeded synthetic inputs for the Gated DeltaNet core.

This module holds the input recipe only -- no arithmetic of the recurrence.
Both the tests (for the CUDA path and for the fp64 oracle) and the benchmark
draw their inputs from here, so the two sides always see the same values.

Recipe (the workloads below):
  * q, k ~ N(0, 1) per element, then L2-normalised per (token, head) in fp32
    and stored in the workload dtype.  The Qwen3.8-Next reading notes
    (jianyuh.github.io, section 2.1, "Feature parameterization") normalise q
    and k before the recurrence and call the normalisation load-bearing; the
    core does not re-normalise.
  * v ~ N(0, 1), stored in the workload dtype.
  * alpha = exp(-softplus(a) * s), a ~ N(0, 1), fp32: the decay gate lies in
    (0, 1) (section 2.1, "Gating dynamics" -- a double-exponential gate with a
    per-head time constant; here exp(A) is folded into the scale s).
  * beta = sigmoid(N(0, 1)), fp32 (section 2.1, beta = sigma(W_beta x)).
  * S0 ~ N(0, s0_std^2) fp32, or absent (zero state) when s0_std == 0.
Every tensor has its own generator seeded from (seed, tensor name), drawn in
the fixed order a, b, q, k, v, S0.

Upstream gradients for the backward pass (no workload of the sources fixes
them): dy ~ N(0, 1) in the workload dtype and dS_T ~ N(0, ds_std^2) fp32
(absent when ds_std == 0), each from its own named generator.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import torch

# Named workloads: shapes and gate scales of the five reference workloads, and a weak-decay variant.
WORKLOADS = {
    # B=1, H=2, T=256, d=64, fp32, gate scale 0.1, zero initial state.
    "tiny": dict(kind="prefill", B=1, T=256, Hqk=2, Hv=2, d=64, dtype="f32", decay_scale=0.1, s0_std=0.0),
    # B=2, H=16, T=4096, d=128, bf16, gate scale 0.05, zero initial state.
    "train": dict(kind="prefill", B=2, T=4096, Hqk=16, Hv=16, d=128, dtype="bf16", decay_scale=0.05, s0_std=0.0),
    # B=1, 16 q/k heads shared by 32 v heads, T=65536, d=128, S0 ~ N(0, 0.02^2).
    "grouped": dict(kind="prefill", B=1, T=65536, Hqk=16, Hv=32, d=128, dtype="bf16", decay_scale=0.05, s0_std=0.02),
    # B=256 sequences, 32 v heads over 16 q/k heads, d=128, 128 single-token steps.
    "decode": dict(kind="decode", B=256, steps=128, Hqk=16, Hv=32, d=128, dtype="bf16", decay_scale=0.05, s0_std=0.02),
    # B=1, H=16, T=2^20, d=128, bf16, gate scale 0.01, zero initial state.
    "long": dict(kind="prefill", B=1, T=1 << 20, Hqk=16, Hv=16, d=128, dtype="bf16", decay_scale=0.01, s0_std=0.0),
    # The grouped shape with gates that barely decay (gate scale 1.2e-4: mean log alpha
    # about -1e-4 per token, alpha ~ 1 - 1e-4), the regime where no short window of
    # preceding tokens forgets the state.
    "weak": dict(kind="prefill", B=1, T=65536, Hqk=16, Hv=32, d=128, dtype="bf16", decay_scale=1.2e-4, s0_std=0.02),
}

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _randn(shape, seed, name, device):
    return torch.randn(shape, generator=_gen(seed, name, device), device=device, dtype=torch.float32)


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)


@dataclass
class PrefillInputs:
    q: torch.Tensor        # [B, T, Hqk, dk]
    k: torch.Tensor        # [B, T, Hqk, dk]
    v: torch.Tensor        # [B, T, Hv, dv]
    alpha: torch.Tensor    # [B, T, Hv] fp32
    beta: torch.Tensor     # [B, T, Hv] fp32
    S0: torch.Tensor | None  # [B, Hv, dk, dv] fp32


def make_prefill_inputs(B, T, Hqk, Hv, d, dtype="bf16", decay_scale=0.05, s0_std=0.0,
                        seed=0, device="cpu", dv=None) -> PrefillInputs:
    dk = d
    dv = d if dv is None else dv
    td = torch_dtype(dtype)
    a = _randn((B, T, Hv), seed, "a", device)
    b = _randn((B, T, Hv), seed, "b", device)
    alpha = torch.exp(-torch.nn.functional.softplus(a) * decay_scale)
    beta = torch.sigmoid(b)
    del a, b
    q = _unit_rows(_randn((B, T, Hqk, dk), seed, "q", device)).to(td)
    k = _unit_rows(_randn((B, T, Hqk, dk), seed, "k", device)).to(td)
    v = _randn((B, T, Hv, dv), seed, "v", device).to(td)
    S0 = None
    if s0_std > 0:
        S0 = _randn((B, Hv, dk, dv), seed, "S0", device) * s0_std
    return PrefillInputs(q.contiguous(), k.contiguous(), v.contiguous(), alpha.contiguous(), beta.contiguous(), S0)


@dataclass
class BackwardGrads:
    dy: torch.Tensor             # [B, T, Hv, dv], workload dtype
    dS_T: torch.Tensor | None    # [B, Hv, dk, dv] fp32


def make_backward_grads(B, T, Hv, d, dtype="bf16", ds_std=1.0, seed=0, device="cpu") -> BackwardGrads:
    dy = _randn((B, T, Hv, d), seed, "dy", device).to(torch_dtype(dtype)).contiguous()
    dS_T = _randn((B, Hv, d, d), seed, "dS_T", device) * ds_std if ds_std > 0 else None
    return BackwardGrads(dy, dS_T)


@dataclass
class DecodeInputs:
    q: torch.Tensor        # [steps, B, 1, Hqk, dk]
    k: torch.Tensor        # [steps, B, 1, Hqk, dk]
    v: torch.Tensor        # [steps, B, 1, Hv, dv]
    alpha: torch.Tensor    # [steps, B, 1, Hv] fp32
    beta: torch.Tensor     # [steps, B, 1, Hv] fp32
    S0: torch.Tensor       # [B, Hv, dk, dv] fp32


def make_decode_inputs(B, steps, Hqk, Hv, d, dtype="bf16", decay_scale=0.05, s0_std=0.02,
                       seed=0, device="cpu") -> DecodeInputs:
    """Fresh q, k, v, alpha, beta for every step; one initial state."""
    x = make_prefill_inputs(steps * B, 1, Hqk, Hv, d, dtype, decay_scale, 0.0, seed, device)
    S0 = _randn((B, Hv, d, d), seed, "S0", device) * s0_std
    sh = lambda t: t.reshape(steps, B, *t.shape[1:])  # noqa: E731
    return DecodeInputs(sh(x.q), sh(x.k), sh(x.v), sh(x.alpha), sh(x.beta), S0.contiguous())


def workload_inputs(name: str, seed: int = 0, device="cpu", **overrides):
    """Inputs of a named workload (optionally with some fields overridden)."""
    w = dict(WORKLOADS[name])
    w.update(overrides)
    kind = w.pop("kind")
    if kind == "decode":
        return make_decode_inputs(w["B"], w["steps"], w["Hqk"], w["Hv"], w["d"], w["dtype"],
                                  w["decay_scale"], w["s0_std"], seed, device)
    return make_prefill_inputs(w["B"], w["T"], w["Hqk"], w["Hv"], w["d"], w["dtype"],
                               w["decay_scale"], w["s0_std"], seed, device)


@dataclass
class LayerInputs:
    xq: torch.Tensor       # [B, T, Hqk, d] bf16: W_q x
    xk: torch.Tensor       # [B, T, Hqk, d] bf16: W_k x
    xv: torch.Tensor       # [B, T, Hv, d]  bf16: W_v x
    wq: torch.Tensor       # [Hqk*d, K] fp32 convolution taps
    wk: torch.Tensor
    wv: torch.Tensor       # [Hv*d, K]
    a_raw: torch.Tensor    # [B, T, Hv] fp32: W_alpha x
    b_raw: torch.Tensor    # [B, T, Hv] fp32: W_beta x
    A: torch.Tensor        # [Hv] fp32
    b_alpha: torch.Tensor  # [Hv] fp32
    state_q: torch.Tensor | None   # [B, K-1, Hqk*d] bf16 incoming convolution states
    state_k: torch.Tensor | None
    state_v: torch.Tensor | None
    y: torch.Tensor        # [B, T, Hv, d] bf16: recurrence output (epilogue input)
    z: torch.Tensor        # [B, T, Hv, d] bf16: W_z x
    norm_w: torch.Tensor   # [d] fp32 zero-centred RMSNorm weight


def make_layer_inputs(B, T, Hqk, Hv, d, kconv=4, decay_scale=0.05, seed=0, device="cpu",
                      with_state=False, vary_heads=False) -> LayerInputs:
    """Inputs of the layer steps around the recurrence.

    Projections (W_q x, ..., W_z x) and y ~ N(0, 1) per element, stored bf16;
    convolution taps ~ N(0, 1/kconv); W_alpha x, W_beta x ~ N(0, 1) fp32;
    norm weight ~ N(0, 0.1^2).  With A = ln(decay_scale) and b_alpha = 0 the
    decay gate exp(-exp(A) softplus(a)) has exactly the distribution of the
    core workloads' alpha (exp(-softplus(a) * decay_scale)); vary_heads adds
    N(0, 0.5^2) per head to both, so per-head indexing is exercised.  Incoming
    convolution states (with_state) ~ N(0, 1) bf16."""
    bf = torch.bfloat16
    xq = _randn((B, T, Hqk, d), seed, "xq", device).to(bf)
    xk = _randn((B, T, Hqk, d), seed, "xk", device).to(bf)
    xv = _randn((B, T, Hv, d), seed, "xv", device).to(bf)
    sc = 1.0 / kconv ** 0.5
    wq = _randn((Hqk * d, kconv), seed, "wq", device) * sc
    wk = _randn((Hqk * d, kconv), seed, "wk", device) * sc
    wv = _randn((Hv * d, kconv), seed, "wv", device) * sc
    a_raw = _randn((B, T, Hv), seed, "a_raw", device)
    b_raw = _randn((B, T, Hv), seed, "b_raw", device)
    A = torch.full((Hv,), float(torch.log(torch.tensor(decay_scale))), device=device)
    b_alpha = torch.zeros(Hv, device=device)
    if vary_heads:
        A = A + 0.5 * _randn((Hv,), seed, "A", device)
        b_alpha = 0.5 * _randn((Hv,), seed, "b_alpha", device)
    st = (lambda H, n: _randn((B, kconv - 1, H * d), seed, n, device).to(bf)) if with_state else (lambda H, n: None)
    y = _randn((B, T, Hv, d), seed, "y", device).to(bf)
    z = _randn((B, T, Hv, d), seed, "z", device).to(bf)
    norm_w = 0.1 * _randn((d,), seed, "norm_w", device)
    return LayerInputs(xq, xk, xv, wq.contiguous(), wk.contiguous(), wv.contiguous(), a_raw, b_raw, A.contiguous(),
                       b_alpha.contiguous(), st(Hqk, "state_q"), st(Hqk, "state_k"), st(Hv, "state_v"), y, z, norm_w)


def make_channelwise_alpha(B, T, Hv, dk, decay_scale=0.05, seed=0, device="cpu") -> torch.Tensor:
    """Channel-wise decay gate [B, T, Hv, dk] fp32: alpha = exp(-softplus(a) * decay_scale),
    a ~ N(0, 1) drawn independently per key channel (the per-channel form of the scalar recipe)."""
    a = _randn((B, T, Hv, dk), seed, "a_cw", device)
    return torch.exp(-torch.nn.functional.softplus(a) * decay_scale).contiguous()
