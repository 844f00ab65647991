"""fp64 oracle for the gradients of the gated delta recurrence (the backward
pass).  Test infrastructure only: the library never imports this module.

The forward map is the four-line recurrence of the Qwen3.8-Next reading notes
(jianyuh.github.io, section 2.1 "Gated DeltaNet"), per (batch, value head),
for t = 1..T:

    S~_t = alpha_t S_{t-1}
    e_t  = v_t - S~_t^T k_t
    S_t  = S~_t + beta_t k_t e_t^T
    y_t  = S_t^T q_t

Given the upstream gradients dy_t = dL/dy_t and dS_T = dL/dS_T, the reverse
pass walks t = T..1 with G = dL/dS_t (starting from dS_T) and applies the
chain rule to each line in reverse order:

    y_t  = S_t^T q_t           dq_t  = S_t dy_t              G += q_t dy_t^T
    S_t  = S~ + b k e^T        db_t  = k_t^T G e_t           dk_t += b_t G e_t
                               de_t  = b_t G^T k_t           G~ = G
    e_t  = v_t - S~^T k_t      dv_t  = de_t                  dk_t -= S~ de_t
                               G~   -= k_t de_t^T
    S~   = a S_{t-1}           da_t  = <G~, S_{t-1}>         G_{t-1} = a_t G~

and dS0 = G_0.  Query/key head hk is shared by the value heads h with
h // (Hv/Hqk) == hk, so dq and dk sum over those heads.  The forward states are
kept (T states of dk x dv per head), so the tensors must be small; this is a
checker, not a training kernel.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def recurrence_grad(q, k, v, alpha, beta, S0, dy, dS_T=None):
    """Gradients of L = sum(dy * y) + sum(dS_T * S_T) with respect to every input.

    Shapes as the forward oracle: q, k [B,T,Hqk,dk]; v, dy [B,T,Hv,dv];
    alpha, beta [B,T,Hv]; S0, dS_T [B,Hv,dk,dv] (None: zeros).  Returns a dict
    with dq, dk, dv, dalpha, dbeta, dS0 (float64) and the forward y, S_T."""
    q, k, v, alpha, beta, S0, dy, dS_T = (_f64(t) for t in (q, k, v, alpha, beta, S0, dy, dS_T))
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    group = Hv // Hqk
    out = {
        "dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
        "dalpha": np.zeros_like(alpha), "dbeta": np.zeros_like(beta),
        "dS0": np.zeros((B, Hv, dk, dv)), "y": np.zeros((B, T, Hv, dv)), "S_T": np.zeros((B, Hv, dk, dv)),
    }
    for b in range(B):
        for h in range(Hv):
            hk = h // group
            S = np.zeros((dk, dv)) if S0 is None else S0[b, h].copy()
            states = [S.copy()]           # states[t] = S_t (S_0 first)
            for t in range(T):
                a, bt = alpha[b, t, h], beta[b, t, h]
                kt, qt, vt = k[b, t, hk], q[b, t, hk], v[b, t, h]
                St = a * S
                e = vt - St.T @ kt
                S = St + bt * np.outer(kt, e)
                out["y"][b, t, h] = S.T @ qt
                states.append(S.copy())
            out["S_T"][b, h] = S
            G = np.zeros((dk, dv)) if dS_T is None else dS_T[b, h].copy()
            for t in range(T - 1, -1, -1):
                a, bt = alpha[b, t, h], beta[b, t, h]
                kt, qt, vt = k[b, t, hk], q[b, t, hk], v[b, t, h]
                Sp = states[t]
                St = a * Sp
                e = vt - St.T @ kt
                S = states[t + 1]
                # y_t = S_t^T q_t
                out["dq"][b, t, hk] += S @ dy[b, t, h]
                G = G + np.outer(qt, dy[b, t, h])
                # S_t = S~ + beta k e^T
                out["dbeta"][b, t, h] = kt @ G @ e
                out["dk"][b, t, hk] += bt * (G @ e)
                de = bt * (G.T @ kt)
                Gt = G.copy()
                # e = v - S~^T k
                out["dv"][b, t, h] = de
                out["dk"][b, t, hk] -= St @ de
                Gt -= np.outer(kt, de)
                # S~ = alpha S_{t-1}
                out["dalpha"][b, t, h] = np.sum(Gt * Sp)
                G = a * Gt
            out["dS0"][b, h] = G
    return out
