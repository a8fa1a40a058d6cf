"""Pins for the blockwise (UT-transform) restatement in ``oracle/chunked.py``:
its chunk factors against explicit products of the transitions, and its full
forward against the literal oracle.

Sources ("PaTH Attention ..." slides): frames "A triangular representation
makes paths computable", "A right-to-left scan accumulates cross-block paths"
and "Backup: fix orientation before implementing UT products".
"""
import numpy as np
import pytest

from oracle import path_oracle_fwd
from oracle.chunked import chunk_factors, path_chunked_fwd, path_chunked_logits


def _chunk(rng, C, d, beta_lo=None):
    W = rng.standard_normal((C, d))
    W /= np.linalg.norm(W, axis=1, keepdims=True)
    K = rng.standard_normal((C, d))
    Q = rng.standard_normal((C, d))
    if beta_lo is None:
        b = 2.0 / (1.0 + np.exp(-rng.standard_normal(C)))
    else:
        b = rng.uniform(beta_lo, 2.0, C)
    return W, K, Q, b


def _prod(H, ts, d):
    P = np.eye(d)
    for t in ts:
        P = P @ H[t]
    return P


@pytest.mark.parametrize("C,d,beta_lo", [(8, 5, None), (16, 6, None), (12, 4, 1.98)])
def test_chunk_factors_match_explicit_products(C, d, beta_lo):
    rng = np.random.default_rng(C * 10 + d)
    W, K, Q, b = _chunk(rng, C, d, beta_lo)
    f = chunk_factors(W, K, Q, b)
    H = [np.eye(d) - b[t] * np.outer(W[t], W[t]) for t in range(C)]
    # H_C ... H_1 = I - W^T U W, and the transition F = H_1 ... H_C
    np.testing.assert_allclose(_prod(H, range(C - 1, -1, -1), d),
                               np.eye(d) - W.T @ f["U"] @ W, atol=1e-12)
    np.testing.assert_allclose(_prod(H, range(C), d), f["F"], atol=1e-12)
    np.testing.assert_allclose(np.eye(d) - f["G"], f["F"].T, atol=1e-12)
    assert np.allclose(np.triu(f["U"], 1), 0.0)
    for i in range(C):
        # left-arrow q_i = H_1 ... H_i q_i
        np.testing.assert_allclose(f["Ql"][i], _prod(H, range(i + 1), d) @ Q[i],
                                   atol=1e-12)
        # right-arrow k_i = H_C ... H_{i+1} k_i
        np.testing.assert_allclose(f["Kr"][i], _prod(H, range(C - 1, i, -1), d) @ K[i],
                                   atol=1e-12)
        for j in range(i + 1):
            assert abs(f["Adiag"][i, j] - K[j] @ _prod(H, range(j + 1, i + 1), d) @ Q[i]) < 1e-11


@pytest.mark.parametrize("T,C,fox", [(37, 4, False), (37, 8, True), (64, 16, False),
                                     (50, 16, True), (1, 8, False), (16, 16, True)])
def test_chunked_forward_matches_literal_oracle(T, C, fox):
    rng = np.random.default_rng(T + C)
    B, H, d = 1, 2, 6
    x = [rng.standard_normal((B, H, T, d)) for _ in range(4)]
    w = x[3] / np.linalg.norm(x[3], axis=-1, keepdims=True)
    b = 2.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T))))
    lf = np.log(1.0 / (1.0 + np.exp(-(2 + rng.standard_normal((B, H, T)))))) if fox else None
    o1, l1 = path_oracle_fwd(x[0], x[1], x[2], w, b, logf=lf)
    o2, l2 = path_chunked_fwd(x[0], x[1], x[2], w, b, C, logf=lf)
    np.testing.assert_allclose(o2, o1, atol=1e-10, rtol=0)
    np.testing.assert_allclose(l2, l1, atol=1e-10, rtol=0)


def test_chunk_size_does_not_change_logits():
    rng = np.random.default_rng(99)
    T, d = 48, 5
    q, k = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    w = rng.standard_normal((T, d))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    b = rng.uniform(1.9, 2.0, T)  # near reflections keep long paths alive
    S4 = path_chunked_logits(q, k, w, b, 4)
    for C in (3, 8, 16, 48, 64):
        S = path_chunked_logits(q, k, w, b, C)
        fin = np.isfinite(S4)
        assert np.array_equal(fin, np.isfinite(S))
        np.testing.assert_allclose(S[fin], S4[fin], atol=1e-11)
