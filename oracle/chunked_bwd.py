"""Blockwise backward of PaTH / PaTH-FoX attention in fp64 numpy -- TEST
INFRASTRUCTURE (the blueprint of a GPU backward, checked against the autograd
oracle in ``oracle/backward.py``).

The forward is the blockwise scan of ``oracle/chunked.py`` ("PaTH Attention:
Position Encoding via Accumulating Householder Transformations", slides,
frames "A triangular representation makes paths computable", "A right-to-left
scan accumulates cross-block paths", "Backup: fix orientation before
implementing UT products").  Per head, with chunks b > c:

    S_bc = scale * X_b^(c) Kr_c^T + gate,   X_b^(b-1) = Ql_b,
    X_b^(c-1) = X_b^(c) F_c^T               (the query crossing chunk c)
    S_bb = scale * Adiag_b + gate           (lower triangle)

The backward, from dS = P * (dP - rowsum(dO * O)):

    dV_c    = sum_b P_bc^T dO_b
    dKr_c   = scale * sum_{b>c} dS_bc^T X_b^(c)
    G_b^(c) = scale * dS_bc Kr_c + G_b^(c-1) F_c        (c = 0 .. b-1, G^(-1) = 0)
    dF_c   += G_b^(c-1)^T X_b^(c)                       (c >= 1)
    dQl_b   = G_b^(b-1),   dAdiag_b = scale * tril(dS_bb)

then, chunk by chunk, through the UT factors (U = (I + L)^{-1} D,
L = strictLower(D W W^T), TK = U strictLower(W K^T), UW = U W,
Ql = Q - tril(Q W^T) UW, Kr = K - TK^T W, F = I - W^T U^T W,
Adiag = tril(Q K^T) - tril(Q W^T) TK) to dQ, dK, dW, dbeta; the gate's
gradient is the reverse cumulative sum of sum_j dS_ij - sum_i dS_ij.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

from .chunked import pad_to_chunks


def _chunk_forward(W, K, Q, beta):
    C = W.shape[0]
    eye = np.eye(C)
    Lm = np.tril((beta[:, None] * W) @ W.T, -1)
    X = solve_triangular(eye + Lm, eye, lower=True)
    U = X * beta[None, :]
    N = np.tril(W @ K.T, -1)
    TK = U @ N
    UW = U @ W
    M = np.tril(Q @ W.T)
    return dict(Lm=Lm, X=X, U=U, N=N, TK=TK, UW=UW, M=M,
                Ql=Q - M @ UW, Kr=K - TK.T @ W,
                F=np.eye(W.shape[1]) - W.T @ U.T @ W,
                Adiag=np.tril(Q @ K.T) - M @ TK)


def _chunk_backward(W, K, Q, beta, f, dQl, dKr, dF, dAdiag):
    """Gradients of one chunk's factors with respect to (Q, K, W, beta)."""
    dQ = dQl.copy()
    dK = dKr.copy()
    dW = np.zeros_like(W)
    # Ql = Q - M UW
    dM = -dQl @ f["UW"].T
    dUW = -f["M"].T @ dQl
    # Kr = K - TK^T W
    dTK = -W @ dKr.T
    dW += -f["TK"] @ dKr
    # F = I - W^T U^T W
    dU = -(W @ dF.T @ W.T)
    dW += -(f["U"] @ W @ dF) - (f["U"].T @ W @ dF.T)
    # Adiag = tril(Q K^T) - M TK   (only the lower triangle is used)
    dA = np.tril(dAdiag)
    dQ += dA @ K
    dK += dA.T @ Q
    dM += -dA @ f["TK"].T
    dTK += -f["M"].T @ dA
    # M = tril(Q W^T)
    dMl = np.tril(dM)
    dQ += dMl @ W
    dW += dMl.T @ Q
    # TK = U N, N = strictLower(W K^T)
    dU += dTK @ f["N"].T
    dN = np.tril(f["U"].T @ dTK, -1)
    dW += dN @ K
    dK += dN.T @ W
    # UW = U W
    dU += dUW @ W.T
    dW += f["U"].T @ dUW
    # U = X diag(beta)
    dX = dU * beta[None, :]
    dbeta = (f["X"] * dU).sum(axis=0)
    # X = (I + Lm)^{-1}: dLm = strictLower(-X^T dX X^T)
    dLm = np.tril(-f["X"].T @ dX @ f["X"].T, -1)
    # Lm_ij = beta_i (w_i . w_j), i > j
    G = W @ W.T
    dbeta += (dLm * G).sum(axis=1)
    dW += (beta[:, None] * dLm) @ W + (beta[:, None] * dLm).T @ W
    return dQ, dK, dW, dbeta


def path_chunked_bwd(q, k, v, w, beta, dout, C, logf=None, scale=None, dlse=None):
    """Gradients (dq, dk, dv, dw, dbeta[, dlogf]) of sum(out * dout)
    (+ sum(lse * dlse)) for one head by the blockwise backward; q, k, v, w:
    [T, d]; beta, logf, dlse: [T].  lse_i = log sum_j exp(S_ij), so its
    gradient adds dlse_i P_ij to dS_ij."""
    q, k, v, w, dout = (np.asarray(x, np.float64) for x in (q, k, v, w, dout))
    beta = np.asarray(beta, np.float64)
    T, d = q.shape
    if scale is None:
        scale = d ** -0.5
    Tp = -(-T // C) * C
    n = Tp // C
    qp, kp, vp, wp, dop = (pad_to_chunks(x, T, C) for x in (q, k, v, w, dout))
    bp = pad_to_chunks(beta, T, C)
    lam = np.cumsum(pad_to_chunks(logf, T, C)) if logf is not None else np.zeros(Tp)
    sl = [slice(c * C, (c + 1) * C) for c in range(n)]
    fac = [_chunk_forward(wp[s], kp[s], qp[s], bp[s]) for s in sl]
    valid = np.arange(Tp) < T
    # forward: logits of every (b, c) pair, exact softmax over real keys
    X = {}
    logits = {}
    for b in range(n):
        Xb = fac[b]["Ql"]
        for c in range(b - 1, -1, -1):
            X[b, c] = Xb
            logits[b, c] = scale * Xb @ fac[c]["Kr"].T
            Xb = Xb @ fac[c]["F"].T
        causal = np.tril(np.ones((C, C), dtype=bool))
        logits[b, b] = np.where(causal, scale * fac[b]["Adiag"], -np.inf)
    S = np.full((Tp, Tp), -np.inf)
    for (b, c), s in logits.items():
        S[sl[b], sl[c]] = s + (lam[sl[b], None] - lam[None, sl[c]])
    S[:, ~valid] = -np.inf
    S[~valid, :] = 0.0
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    P /= P.sum(axis=1, keepdims=True)
    P[~valid, :] = 0.0
    O = P @ vp
    dP = dop @ vp.T
    Dr = (dop * O).sum(axis=1, keepdims=True)
    if dlse is not None:
        Dr = Dr - pad_to_chunks(np.asarray(dlse, np.float64), T, C)[:, None]
    dS = P * (dP - Dr)                       # gradient of the log-weights
    dv = P.T @ dop
    # attention side
    dKr = [np.zeros((C, d)) for _ in range(n)]
    dQl = [np.zeros((C, d)) for _ in range(n)]
    dF = [np.zeros((d, d)) for _ in range(n)]
    dAd = [scale * np.tril(dS[sl[b], sl[b]]) for b in range(n)]
    for b in range(n):
        Gprev = None
        for c in range(b):
            dSbc = dS[sl[b], sl[c]]
            dKr[c] += scale * dSbc.T @ X[b, c]
            G = scale * dSbc @ fac[c]["Kr"]
            if Gprev is not None:
                dF[c] += Gprev.T @ X[b, c]
                G = G + Gprev @ fac[c]["F"]
            Gprev = G
        if b > 0:
            dQl[b] = Gprev
    # chunk side
    dq, dk, dw = (np.zeros((Tp, d)) for _ in range(3))
    db = np.zeros(Tp)
    for c in range(n):
        gQ, gK, gW, gb = _chunk_backward(wp[sl[c]], kp[sl[c]], qp[sl[c]], bp[sl[c]], fac[c],
                                         dQl[c], dKr[c], dF[c], dAd[c])
        dq[sl[c]], dk[sl[c]], dw[sl[c]], db[sl[c]] = gQ, gK, gW, gb
    out = [dq[:T], dk[:T], dv[:T], dw[:T], db[:T]]
    if logf is not None:
        dlam = dS.sum(axis=1) - dS.sum(axis=0)
        out.append(np.cumsum(dlam[::-1])[::-1][:T])
    return tuple(out)
