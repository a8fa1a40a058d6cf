"""Pins for the w / beta producer oracle (``oracle/producer.py``): each step
against a library routine or a property the pages fix, so that a reversed
convolution tap, a wrong normalization axis or a missing factor 2 fails.

Source: "PaTH Attention: Position Encoding via Accumulating Householder
Transformations" (slides, frame "PaTH inserts a learned transformation along
every path"); OpenReview discussion, section "Model Architecture Details".
"""
import numpy as np
import pytest
from scipy.special import expit

from oracle.producer import (beta_gate, l2norm_heads, lowrank_projection, producer_fwd,
                             short_conv)


def _weights(rng, Dm, R, H, d):
    return (rng.standard_normal((R, Dm)) / np.sqrt(Dm), rng.standard_normal((H * d, R)) / np.sqrt(R),
            rng.standard_normal((H * d, 3)), rng.standard_normal((H, Dm)) / np.sqrt(Dm),
            rng.standard_normal(H))


def test_short_conv_is_causal_convolution_per_channel():
    rng = np.random.default_rng(51)
    B, T, Cc = 2, 37, 5
    p = rng.standard_normal((B, T, Cc))
    cw = rng.standard_normal((Cc, 3))
    z = short_conv(p, cw)
    for b in range(B):
        for c in range(Cc):
            # z_t = sum_s h[s] p_{t-s} with h = (cw[c,2], cw[c,1], cw[c,0])
            ref = np.convolve(p[b, :, c], cw[c, ::-1])[:T]
            np.testing.assert_allclose(z[b, :, c], ref, atol=1e-13)


def test_l2norm_per_head():
    rng = np.random.default_rng(52)
    B, T, H, d = 2, 9, 3, 4
    z = rng.standard_normal((B, T, H * d))
    z[0, 3, d:2 * d] = 0.0                      # a zero head vector stays zero
    w = l2norm_heads(z, H, d)
    zz = z.reshape(B, T, H, d).transpose(0, 2, 1, 3)
    n = np.linalg.norm(w, axis=-1)
    mask = np.ones_like(n, dtype=bool)
    mask[0, 1, 3] = False
    np.testing.assert_allclose(n[mask], 1.0, atol=1e-14)
    assert np.all(w[0, 1, 3] == 0.0)
    # same direction as z, per head
    cos = (w * zz).sum(-1)[mask] / np.linalg.norm(zz, axis=-1)[mask]
    np.testing.assert_allclose(cos, 1.0, atol=1e-14)


def test_beta_gate_is_twice_the_logistic():
    rng = np.random.default_rng(53)
    x = rng.standard_normal((2, 7, 6))
    Ub = rng.standard_normal((3, 6))
    bb = rng.standard_normal(3)
    beta = beta_gate(x, Ub, bb)
    ref = 2.0 * expit(np.einsum("btm,hm->bht", x, Ub) + bb[None, :, None])
    np.testing.assert_allclose(beta, ref, atol=1e-15)
    assert np.all((beta > 0) & (beta < 2))
    assert abs(beta_gate(np.zeros((1, 1, 6)), Ub, np.zeros(3))[0, 0, 0] - 1.0) < 1e-15


def test_lowrank_projection_is_the_rank_r_map():
    rng = np.random.default_rng(54)
    x = rng.standard_normal((2, 5, 12))
    Wd, Wu = rng.standard_normal((3, 12)), rng.standard_normal((8, 3))
    p = lowrank_projection(x, Wd, Wu)
    np.testing.assert_allclose(p, np.einsum("btm,cm->btc", x, Wu @ Wd), atol=1e-12)
    assert np.linalg.matrix_rank(p.reshape(-1, 8)) <= 3


@pytest.mark.parametrize("t0", [0, 5, 20])
def test_w_at_t_depends_only_on_tokens_t_minus_2_to_t(t0):
    rng = np.random.default_rng(55)
    B, T, Dm, R, H, d = 1, 24, 16, 4, 2, 4
    Wd, Wu, cw, Ub, bb = _weights(rng, Dm, R, H, d)
    x = rng.standard_normal((B, T, Dm))
    w0, b0 = producer_fwd(x, Wd, Wu, cw, Ub, bb, H, d)
    x2 = x.copy()
    x2[:, t0] += rng.standard_normal(Dm)
    w1, b1 = producer_fwd(x2, Wd, Wu, cw, Ub, bb, H, d)
    changed = np.abs(w1 - w0).max(axis=(0, 1, 3)) > 1e-12
    assert set(np.nonzero(changed)[0]) == {t for t in (t0, t0 + 1, t0 + 2) if t < T}
    bchanged = np.abs(b1 - b0).max(axis=(0, 1)) > 1e-14
    assert set(np.nonzero(bchanged)[0]) == {t0}


def test_identity_taps_reduce_to_normalized_projection():
    rng = np.random.default_rng(56)
    B, T, Dm, R, H, d = 2, 6, 10, 3, 2, 5
    Wd, Wu, _, Ub, bb = _weights(rng, Dm, R, H, d)
    cw = np.tile([0.0, 0.0, 1.0], (H * d, 1))
    x = rng.standard_normal((B, T, Dm))
    w, _ = producer_fwd(x, Wd, Wu, cw, Ub, bb, H, d)
    p = np.einsum("btm,cm->btc", x, Wu @ Wd).reshape(B, T, H, d)
    ref = (p / np.linalg.norm(p, axis=-1, keepdims=True)).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(w, ref, atol=1e-13)
