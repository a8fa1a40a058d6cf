"""CPU oracle for the producer of PaTH's w and beta -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this module.

Written from "PaTH Attention: Position Encoding via Accumulating Householder
Transformations" (slides, frame "PaTH inserts a learned transformation along
every path": w_t from a low-rank projection, a width-3 convolution and an L2
normalization; beta_t = 2 sigmoid(u^T x_t + b)) and the OpenReview discussion
(section "Model Architecture Details": linear projection, short convolution,
L2 normalization per head; low-rank projections in the spirit of LoRA).

Readings where the pages are silent (also listed in the design notes):
  * the low-rank projection is x Wd^T Wu^T with Wd: [R, Dm], Wu: [H*d, R]
    (no bias);
  * the short convolution is causal and depthwise over time, per channel c:
    z_t[c] = cw[c,0] p_{t-2}[c] + cw[c,1] p_{t-1}[c] + cw[c,2] p_t[c], with
    p_s = 0 before the sequence start; no bias, no activation;
  * the L2 normalization is per (token, head) over d: w = z / max(|z|, 1e-12);
  * beta has one row of U ([H, Dm]) and one bias per head.
Everything in fp64 numpy, steps in the pages' order.
"""
from __future__ import annotations

import numpy as np

NORM_FLOOR = 1e-12


def lowrank_projection(x, Wd, Wu):
    """p = (x Wd^T) Wu^T: [B, T, Dm] -> [B, T, H*d]."""
    return (np.asarray(x, np.float64) @ np.asarray(Wd, np.float64).T) @ np.asarray(Wu, np.float64).T


def short_conv(p, cw):
    """Causal width-3 depthwise convolution over time of p [B, T, Cc] with
    taps cw [Cc, 3]: z_t = cw[:,0] p_{t-2} + cw[:,1] p_{t-1} + cw[:,2] p_t."""
    p, cw = np.asarray(p, np.float64), np.asarray(cw, np.float64)
    z = np.zeros_like(p)
    for tap in range(3):
        shift = 2 - tap
        if shift == 0:
            z += cw[:, tap] * p
        else:
            z[:, shift:, :] += cw[:, tap] * p[:, :-shift, :]
    return z


def l2norm_heads(z, H, d):
    """[B, T, H*d] -> [B, H, T, d], each (token, head) vector divided by
    max(|z|, NORM_FLOOR)."""
    B, T, _ = z.shape
    z = np.asarray(z, np.float64).reshape(B, T, H, d)
    nrm = np.sqrt((z * z).sum(axis=-1, keepdims=True))
    return (z / np.maximum(nrm, NORM_FLOOR)).transpose(0, 2, 1, 3).copy()


def beta_gate(x, Ub, bb):
    """beta [B, H, T] = 2 sigmoid(x Ub^T + bb)."""
    a = np.asarray(x, np.float64) @ np.asarray(Ub, np.float64).T + np.asarray(bb, np.float64)
    return (2.0 / (1.0 + np.exp(-a))).transpose(0, 2, 1).copy()


def producer_fwd(x, Wd, Wu, cw, Ub, bb, H, d):
    """x: [B, T, Dm]; Wd: [R, Dm]; Wu: [H*d, R]; cw: [H*d, 3]; Ub: [H, Dm];
    bb: [H].  Returns (w [B, H, T, d], beta [B, H, T]) in fp64: projection,
    convolution, per-head normalization, and the beta gate."""
    p = lowrank_projection(x, Wd, Wu)
    z = short_conv(p, cw)
    return l2norm_heads(z, H, d), beta_gate(x, Ub, bb)
