"""The chunked (WY/UT) form of the backward pass, checked against the fp64
backward oracle on CPU.

This is the algebra a tensor-core backward computes, written in the
convention of the chunked forward: per chunk of C tokens with entering
state S,

    g = cumsum(log alpha), gam = e^g, M_ij = e^(g_i - g_j) (j <= i)
    A = diag(beta) strict(M o K K^T),  T = (I + A)^-1
    W = T diag(beta gam) K,  Ut = T diag(beta) V,  U = Ut - W S  (rows beta_i e_i)
    Y = diag(gam) Q S + (M o Q K^T) U
    S' = gam_last S + (diag(lam) K)^T U,  lam_j = e^(g_last - g_j)

(the gated delta recurrence of the Qwen3.8-Next reading notes, section 2.1,
"Gated DeltaNet", unrolled over a chunk).  The reverse pass over chunks
carries dS, the gradient of the entering state:

    dU = (M o Q K^T)^T dY + diag(lam) K dS'
    dS = gam_last dS' + Q^T diag(gam) dY - W^T dU

which is the serial part, two d x d-sized products per chunk like the
forward's state scan.  Everything else (dQ, dK, dV, dbeta, dlog alpha)
follows per chunk in parallel from S, dS' and the chunk's inputs.  The test
pins that every term matches the token-by-token oracle to rounding, for
ragged and whole chunks.
"""
import numpy as np
import pytest

import oracle.backward as BW


def chunk_fwd(Q, K, V, la, b, S):
    C = Q.shape[0]
    g = np.cumsum(la); gam = np.exp(g)
    Mi = np.tril(np.exp(g[:, None] - g[None, :]))          # j <= i
    Ms = np.tril(Mi, -1)                                    # j < i
    A = b[:, None] * (Ms * (K @ K.T))
    T = np.linalg.inv(np.eye(C) + A)
    W = T @ ((b * gam)[:, None] * K)
    Ut = T @ (b[:, None] * V)
    U = Ut - W @ S
    P = Mi * (Q @ K.T)
    Y = gam[:, None] * (Q @ S) + P @ U
    lam = np.exp(g[-1] - g)
    Sn = gam[-1] * S + (lam[:, None] * K).T @ U
    return dict(g=g, gam=gam, Mi=Mi, Ms=Ms, A=A, T=T, W=W, Ut=Ut, U=U, P=P, Y=Y, lam=lam, Sn=Sn)

def chunk_bwd(Q, K, V, la, b, S, f, dY, dSn):
    """Gradients of <dY, Y> + <dSn, S'> for one chunk: dQ, dK, dV, dla (d log alpha), db, dS."""
    g, gam, Mi, Ms, T, W, U, P, lam = (f[k] for k in ('g', 'gam', 'Mi', 'Ms', 'T', 'W', 'U', 'P', 'lam'))
    dg = np.zeros_like(g)
    # S' = gam_last S + Kb^T U
    dU = lam[:, None] * (K @ dSn)                       # Kb dS'
    dS = gam[-1] * dSn
    dg[-1] += gam[-1] * np.sum(dSn * S)
    dlam = np.sum((K @ dSn) * U, axis=1)                # d lam_j = k_j^T dS' u_j
    dK = lam[:, None] * (U @ dSn.T)
    # lam_j = e^{g_last - g_j}
    dg[-1] += np.sum(dlam * lam); dg -= dlam * lam
    # Y = diag(gam) Q S + P U
    dU += P.T @ dY
    dS += Q.T @ (gam[:, None] * dY)
    QS = Q @ S
    dQ = gam[:, None] * (dY @ S.T)
    dg += gam * np.sum(dY * QS, axis=1)
    dP = dY @ U.T                                       # only j <= i used
    dQK = dP * Mi                                       # d(QK^T)
    dQ += dQK @ K
    dK += dQK.T @ Q
    dMi = dP * (Q @ K.T) * Mi                           # d g via M_ij = e^{g_i - g_j}
    dg += dMi.sum(1); dg -= dMi.sum(0)
    # U = Ut - W S
    dUt = dU
    dW = -dU @ S.T
    dS -= W.T @ dU
    # W = T diag(b gam) K, Ut = T diag(b) V
    bg = b * gam
    TtdW = T.T @ dW; TtdUt = T.T @ dUt
    dK += bg[:, None] * TtdW
    dV = b[:, None] * TtdUt
    db = gam * np.sum(TtdW * K, axis=1) + np.sum(TtdUt * V, axis=1)
    dg += b * gam * np.sum(TtdW * K, axis=1)
    dT = dW @ (bg[:, None] * K).T + dUt @ (b[:, None] * V).T
    # T = (I + A)^-1  ->  dA = -T^T dT T^T
    dA = -T.T @ dT @ T.T
    dA = np.tril(dA, -1)
    # A = diag(b) (Ms o KK^T)
    KK = K @ K.T
    db += np.sum(dA * Ms * KK, axis=1)
    dKK = dA * b[:, None] * Ms
    dK += (dKK + dKK.T) @ K
    dMs = dA * b[:, None] * KK * Ms
    dg += dMs.sum(1); dg -= dMs.sum(0)
    # g = cumsum(la): dla_r = sum_{i >= r} dg_i
    dla = np.cumsum(dg[::-1])[::-1]
    return dQ, dK, dV, dla, db, dS

def chunked_grad(q, k, v, a, b, S0, dy, dST, C):
    """One head: q, k [T, dk]; v, dy [T, dv]; a, b [T]; S0, dST [dk, dv]."""
    T = q.shape[0]; la = np.log(a)
    bounds = [(c, min(c + C, T)) for c in range(0, T, C)]
    Ss = [S0]; fs = []
    for (c0, c1) in bounds:                              # forward: entering states per chunk
        f = chunk_fwd(q[c0:c1], k[c0:c1], v[c0:c1], la[c0:c1], b[c0:c1], Ss[-1])
        fs.append(f); Ss.append(f['Sn'])
    out = {n: np.zeros_like(x) for n, x in (('dq', q), ('dk', k), ('dv', v), ('dla', a), ('db', b))}
    dS = dST.copy()
    for ci in range(len(bounds) - 1, -1, -1):           # reverse scan over chunks
        c0, c1 = bounds[ci]
        dQ, dK, dV, dla, db, dS = chunk_bwd(q[c0:c1], k[c0:c1], v[c0:c1], la[c0:c1], b[c0:c1], Ss[ci], fs[ci],
                                            dy[c0:c1], dS)
        out['dq'][c0:c1] = dQ; out['dk'][c0:c1] = dK; out['dv'][c0:c1] = dV
        out['dla'][c0:c1] = dla; out['db'][c0:c1] = db
    out['dS0'] = dS
    out['y'] = np.concatenate([f['Y'] for f in fs]); out['S_T'] = Ss[-1]
    return out


@pytest.mark.parametrize("T,d,C", [(37, 8, 8), (64, 16, 16), (50, 12, 64), (9, 4, 4), (1, 6, 64)])
def test_chunked_backward_matches_oracle(T, d, C):
    rng = np.random.default_rng(T * 100 + d)
    q = rng.standard_normal((T, d))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k = rng.standard_normal((T, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, d))
    a = rng.uniform(0.6, 1.0, T)
    b = rng.uniform(0.05, 0.95, T)
    S0 = 0.3 * rng.standard_normal((d, d))
    dy = rng.standard_normal((T, d))
    dST = rng.standard_normal((d, d))
    m = chunked_grad(q, k, v, a, b, S0, dy, dST, C)
    one = lambda x: x[None, :, None]  # noqa: E731
    o = BW.recurrence_grad(one(q), one(k), one(v), one(a), one(b), S0[None, None], one(dy), dST[None, None])
    ref = dict(dq=o["dq"][0, :, 0], dk=o["dk"][0, :, 0], dv=o["dv"][0, :, 0], dla=a * o["dalpha"][0, :, 0],
               db=o["dbeta"][0, :, 0], dS0=o["dS0"][0, 0], y=o["y"][0, :, 0], S_T=o["S_T"][0, 0])
    for n in ref:
        assert np.abs(m[n] - ref[n]).max() <= 1e-12 * max(1.0, np.abs(ref[n]).max()), n
