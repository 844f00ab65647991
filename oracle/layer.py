"""fp64 oracle for the GDN layer's steps on either side of the recurrence.

Test infrastructure only: the library never imports this module.

The Qwen3.8-Next reading notes (jianyuh.github.io, section 2.1 "Gated
DeltaNet") give the feature parameterisation around the recurrence:
  * "Feature parameterization": q_t = L2Norm(SiLU(ShortConv(W_q x_t))),
    k_t = L2Norm(SiLU(ShortConv(W_k x_t))), v_t = SiLU(ShortConv(W_v x_t)),
    the convolutions being short, causal and depthwise ("Inside GDN": "short
    depthwise causal convolutions");
  * "Gating dynamics": beta_t = sigma(W_beta x_t) and
    alpha_t = exp[-exp(A) * softplus(W_alpha x_t + b_alpha)], with a per-head
    constant A;
  * the output o_t = W_o[sigma(W_z x_t) * RMSNorm(y_t)], the RMSNorm being
    zero-centred.
The projections W_* x_t are inputs here (plain GEMMs outside this step); the
functions below take them as given and compute everything in between, in
fp64, from the stored input values.

Readings where the pages are silent (each listed in the design notes):
  * ShortConv: per channel c, out[t, c] = sum_{i<K} w[c, i] * x[t-K+1+i, c],
    no bias; tap K-1 multiplies the current token.  The K-1 inputs before the
    first token come from a carried convolution state (zeros for a fresh
    sequence), and the last K-1 inputs are returned as the next state.
  * L2Norm(u) = u / sqrt(sum(u^2) + eps) over the head dimension, eps = 1e-6.
  * RMSNorm(y) = y / sqrt(mean(y^2) + eps) * (1 + w) over the head dimension:
    "zero-centred" read as a learned weight stored as its offset from 1, one
    weight vector shared by the heads, eps = 1e-6.
  * softplus(u) = log(1 + e^u).
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6
RMS_EPS = 1e-6


def f64(x):
    """Exact upcast of a numpy array or torch tensor to float64."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def short_conv(x, w, state=None):
    """Causal depthwise convolution along time.

    x: [B, T, C]; w: [C, K] (tap K-1 multiplies the current token);
    state: [B, K-1, C], the K-1 inputs preceding token 0 (None: zeros).
    Returns (out [B, T, C], state_out [B, K-1, C]: the last K-1 inputs)."""
    x, w = f64(x), f64(w)
    B, T, C = x.shape
    K = w.shape[1]
    prev = np.zeros((B, K - 1, C)) if state is None else f64(state)
    xp = np.concatenate([prev, x], axis=1)          # [B, K-1+T, C]
    out = np.zeros((B, T, C))
    for i in range(K):
        out += w[:, i] * xp[:, i:i + T, :]
    return out, xp[:, T:, :].copy()


def silu(u):
    u = f64(u)
    return u / (1.0 + np.exp(-u))


def sigmoid(u):
    u = f64(u)
    return 1.0 / (1.0 + np.exp(-u))


def softplus(u):
    u = f64(u)
    return np.where(u > 0, u + np.log1p(np.exp(-np.abs(u))), np.log1p(np.exp(u)))


def l2norm(u, eps=L2_EPS):
    """u / sqrt(sum(u^2) + eps) over the last axis."""
    u = f64(u)
    return u / np.sqrt(np.sum(u * u, axis=-1, keepdims=True) + eps)


def rmsnorm_zc(y, w, eps=RMS_EPS):
    """Zero-centred RMSNorm over the last axis: y / sqrt(mean(y^2) + eps) * (1 + w)."""
    y, w = f64(y), f64(w)
    return y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + eps) * (1.0 + w)


def gates(a_raw, b_raw, A, b_alpha):
    """alpha = exp(-exp(A_h) * softplus(a + b_alpha_h)), beta = sigma(b): [B, T, Hv] each."""
    a_raw, b_raw, A, b_alpha = f64(a_raw), f64(b_raw), f64(A), f64(b_alpha)
    alpha = np.exp(-np.exp(A) * softplus(a_raw + b_alpha))
    beta = sigmoid(b_raw)
    return alpha, beta


def feature(x, w, state=None, normalise=True, eps=L2_EPS):
    """One of q, k (normalise=True) or v (False) from its projection x [B, T, H, d].

    Returns (feature [B, T, H, d], conv state out [B, K-1, H*d])."""
    x = f64(x)
    B, T, H, d = x.shape
    c, st = short_conv(x.reshape(B, T, H * d), w, state)
    u = silu(c).reshape(B, T, H, d)
    return (l2norm(u, eps) if normalise else u), st


def prologue(xq, xk, xv, wq, wk, wv, a_raw, b_raw, A, b_alpha, state_q=None, state_k=None, state_v=None):
    """Everything between the input projections and the recurrence."""
    q, sq = feature(xq, wq, state_q, True)
    k, sk = feature(xk, wk, state_k, True)
    v, sv = feature(xv, wv, state_v, False)
    alpha, beta = gates(a_raw, b_raw, A, b_alpha)
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, state_q=sq, state_k=sk, state_v=sv)


def epilogue(y, z, w_norm, eps=RMS_EPS):
    """Everything between the recurrence and the output projection:
    sigma(z) * RMSNorm(y), per (token, value head) over dv."""
    return sigmoid(z) * rmsnorm_zc(y, w_norm, eps)
