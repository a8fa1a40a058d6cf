"""GPU parity of the w / beta producer (``path_producer_fwd``) against the
fp64 oracle in ``oracle/producer.py``.  Tolerances: fp32 inputs 2e-5 max-abs
on w and beta; bf16 inputs 4e-3 max-abs on w (its bf16 rounding is 2^-9 of a
unit vector's entries) and 2e-5 on beta (fp32 out of bf16 operands).
"""
import numpy as np
import pytest
import torch

import householder_softmax_attention_gb300 as pa
from oracle.producer import producer_fwd
from seeded_inputs import PRODUCER_WORKLOADS, ProducerWorkload, make_producer_inputs

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _run(x):
    dev = {k: v.cuda() for k, v in x.items()}
    H = dev["Ub"].shape[0]
    d = dev["Wu"].shape[0] // H
    w, beta = pa.path_producer_fwd(dev["x"], dev["Wd"], dev["Wu"], dev["cw"], dev["Ub"], dev["bb"],
                                   H, d)
    torch.cuda.synchronize()
    return w, beta, H, d


def _tol(dtype):
    return (4e-3, 2e-5) if dtype == "bf16" else (2e-5, 2e-5)


@pytest.mark.parametrize("wl", [
    ProducerWorkload("p_f32", 2, 150, 128, 2, 64, 16, "f32", seed=1),
    ProducerWorkload("p_f32_d128", 1, 230, 192, 2, 128, 32, "f32", seed=2),
    ProducerWorkload("p_bf16", 3, 150, 256, 4, 128, 64, "bf16", seed=3),
    ProducerWorkload("p_bf16_d64", 2, 333, 512, 8, 64, 48, "bf16", seed=4),
    ProducerWorkload("p_bf16_short", 4, 1, 64, 8, 64, 16, "bf16", seed=5),
    ProducerWorkload("p_bf16_d64_r64", 3, 150, 128, 8, 64, 64, "bf16", seed=6),
    ProducerWorkload("p_bf16_t1_r64", 5, 1, 64, 4, 128, 64, "bf16", seed=7),
    ProducerWorkload("p_bf16_r64_h3", 2, 260, 192, 3, 128, 64, "bf16", seed=8),
], ids=lambda w: w.name)
def test_producer_matches_oracle(wl):
    x = make_producer_inputs(wl)
    w, beta, H, d = _run(x)
    ref_w, ref_b = producer_fwd(*(_np(x[n]) for n in ("x", "Wd", "Wu", "cw", "Ub", "bb")), H, d)
    tw, tb = _tol(wl.dtype)
    assert np.abs(_np(w) - ref_w).max() <= tw
    assert np.abs(_np(beta) - ref_b).max() <= tb
    # the outputs feed the forward directly: unit w per (token, head)
    np.testing.assert_allclose(np.linalg.norm(_np(w), axis=-1), 1.0, atol=2 * tw * np.sqrt(d))


@pytest.mark.parametrize("name", sorted(PRODUCER_WORKLOADS))
def test_full_size_producer_sampled(name):
    """The full workload on the GPU; the oracle recomputes sampled tokens from
    their three-token window (w_t depends on x_{t-2..t} only)."""
    wl = PRODUCER_WORKLOADS[name]
    x = make_producer_inputs(wl, device="cuda")
    w, beta = pa.path_producer_fwd(x["x"], x["Wd"], x["Wu"], x["cw"], x["Ub"], x["bb"], wl.H, wl.d)
    torch.cuda.synchronize()
    g = np.random.default_rng(9)
    picks = [(0, 0), (0, 1), (0, 2), (wl.B - 1, wl.T - 1), (1, 111), (1, 112), (1, 113)]
    picks += [(int(g.integers(wl.B)), int(g.integers(wl.T))) for _ in range(12)]
    W = {n: _np(x[n]) for n in ("Wd", "Wu", "cw", "Ub", "bb")}
    tw, tb = _tol(wl.dtype)
    for b, t in picks:
        t0 = max(0, t - 2)
        xw = _np(x["x"][b:b + 1, t0:t + 1])
        ref_w, ref_b = producer_fwd(xw, W["Wd"], W["Wu"], W["cw"], W["Ub"], W["bb"], wl.H, wl.d)
        assert np.abs(_np(w[b, :, t]) - ref_w[0, :, -1]).max() <= tw, (b, t)
        assert np.abs(_np(beta[b, :, t]) - ref_b[0, :, -1]).max() <= tb, (b, t)

