"""Blockwise (UT-transform) formulation of PaTH attention in fp64 numpy --
TEST INFRASTRUCTURE.

Written from "PaTH Attention: Position Encoding via Accumulating Householder
Transformations" (discussion slides for arXiv:2505.16381v2):

* frame "A triangular representation makes paths computable":
  with the chunk's ``w_t^T`` stacked as rows of ``W`` and ``D = diag(beta)``,
  ``U = (I + strictLower(D W W^T))^{-1} D`` and ``H_L ... H_1 = I - W^T U W``;
  intra-chunk logits ``lower(Q K^T) - lower(Q W^T) U strictLower(W K^T)``.
* frame "Backup: fix orientation before implementing UT products":
  boundary-adjusted queries ``Q - lower(Q W^T) U W`` (``q_i`` carried through
  ``H_i .. H_first``), keys ``K - (U strictLower(W K^T))^T W`` (``k_j`` carried
  through ``H_{j+1} .. H_last``) and the chunk transition
  ``F = H_first ... H_last = I - W^T U^T W``.
* frame "A right-to-left scan accumulates cross-block paths":
  diagonal chunk first, then for ``c = b-1 .. 0`` the logits
  ``Q_work K_c^T`` followed by ``Q_work <- Q_work F_c^T``.

A chunk that the sequence does not fill is padded with ``beta = 0`` tokens
(``H = I``), which leaves every real logit unchanged.

This module shares nothing with the literal oracle in ``path_oracle.c``; the
two are checked against each other in the tests.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def chunk_factors(W, K, Q, beta):
    """Factors of one chunk (all ``[C, d]`` except ``beta`` ``[C]``).

    Returns a dict with
      U    -- ``(I + strictLower(D W W^T))^{-1} D`` (lower triangular, C x C)
      UW   -- ``U W``
      TK   -- ``U strictLower(W K^T)``
      Kr   -- boundary-adjusted keys ``K - TK^T W``      (right arrow K)
      Ql   -- boundary-adjusted queries ``Q - lower(Q W^T) U W``  (left arrow Q)
      F    -- ``H_first ... H_last = I - W^T U^T W``
      G    -- ``W^T U W`` so that ``q^T F^T = q^T - q^T G``
      Adiag -- intra-chunk logits ``lower(Q K^T) - lower(Q W^T) TK``
               (entries above the diagonal are 0, not masked here)
    """
    W, K, Q = (np.asarray(x, dtype=np.float64) for x in (W, K, Q))
    beta = np.asarray(beta, dtype=np.float64)
    C, d = W.shape
    eye = np.eye(C)
    D = np.diag(beta)
    Lmat = np.tril(D @ W @ W.T, -1)
    U = solve_triangular(eye + Lmat, D, lower=True)
    UW = U @ W
    TK = U @ np.tril(W @ K.T, -1)
    Kr = K - TK.T @ W
    QWl = np.tril(Q @ W.T)
    Ql = Q - QWl @ UW
    F = np.eye(d) - W.T @ U.T @ W
    G = W.T @ UW
    Adiag = np.tril(Q @ K.T) - QWl @ TK
    return dict(U=U, UW=UW, TK=TK, Kr=Kr, Ql=Ql, F=F, G=G, Adiag=Adiag)


def pad_to_chunks(x, T, C, axis=0):
    """Zero-pad axis ``axis`` (length T) up to a multiple of C."""
    Tp = -(-T // C) * C
    if Tp == T:
        return np.asarray(x, dtype=np.float64)
    pad = [(0, 0)] * np.ndim(x)
    pad[axis] = (0, Tp - T)
    return np.pad(np.asarray(x, dtype=np.float64), pad)


def head_chunk_factors(q, k, w, beta, C):
    """Factors of every chunk of one head (``q, k, w: [T, d]``), padded."""
    T, d = np.shape(q)
    qp, kp, wp = (pad_to_chunks(x, T, C) for x in (q, k, w))
    bp = pad_to_chunks(beta, T, C)
    n = qp.shape[0] // C
    return [chunk_factors(wp[c * C:(c + 1) * C], kp[c * C:(c + 1) * C],
                          qp[c * C:(c + 1) * C], bp[c * C:(c + 1) * C])
            for c in range(n)]


def path_chunked_logits(q, k, w, beta, C, logf=None, scale=None):
    """``[T, T]`` log-weights of one head by the blockwise scan; entries with
    ``j > i`` are ``-inf``.  ``scale`` multiplies only the PaTH logit; the
    gate ``sum_{s=j+1}^{i} log f_s`` is added outside it."""
    q = np.asarray(q, dtype=np.float64)
    T, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    fac = head_chunk_factors(q, k, w, beta, C)
    n = len(fac)
    Tp = n * C
    A = np.full((Tp, Tp), -np.inf)
    for b in range(n):
        rb = slice(b * C, (b + 1) * C)
        A[rb, rb] = np.where(np.tril(np.ones((C, C), dtype=bool)),
                             fac[b]["Adiag"], -np.inf)
        Qw = fac[b]["Ql"]
        for c in range(b - 1, -1, -1):
            A[rb, c * C:(c + 1) * C] = Qw @ fac[c]["Kr"].T
            Qw = Qw @ fac[c]["F"].T
    A = A[:T, :T]
    S = np.where(np.isfinite(A), scale * A, -np.inf)
    if logf is not None:
        lam = np.cumsum(np.asarray(logf, dtype=np.float64))
        gate = lam[:, None] - lam[None, :]
        S = np.where(np.isfinite(S), S + gate, -np.inf)
    return S


def path_chunked_fwd(q, k, v, w, beta, C, logf=None, scale=None):
    """Forward for ``[..., T, d]`` inputs via the blockwise scan (small T)."""
    q, k, v, w = (np.asarray(x, dtype=np.float64) for x in (q, k, v, w))
    beta = np.asarray(beta, dtype=np.float64)
    *lead, T, d = q.shape
    BH = int(np.prod(lead)) if lead else 1
    qf, kf, vf, wf = (x.reshape(BH, T, d) for x in (q, k, v, w))
    bf = beta.reshape(BH, T)
    lf = None if logf is None else np.asarray(logf, np.float64).reshape(BH, T)
    out = np.zeros((BH, T, d))
    lse = np.zeros((BH, T))
    for h in range(BH):
        S = path_chunked_logits(qf[h], kf[h], wf[h], bf[h], C,
                                None if lf is None else lf[h], scale)
        m = S.max(axis=1, keepdims=True)
        P = np.exp(S - m)
        l = P.sum(axis=1, keepdims=True)
        out[h] = (P @ vf[h]) / l
        lse[h] = (m + np.log(l))[:, 0]
    return out.reshape(q.shape), lse.reshape(beta.shape)
