"""GPU parity of the backward pass (path_attn_bwd) against the fp64 blockwise
backward of the oracle (``oracle/chunked_bwd.py``, pinned to the autograd
gradient oracle, itself pinned to finite differences), at sizes that span
several chunks with a ragged tail, plus identities that hold at any size.

Tolerances, per gradient, against the oracle run on the same stored inputs:
  fp32  max-abs <= 1e-4 * max(1, max|ref|)  (the forward's fp32 bar, scaled to
        the gradient's magnitude)
  bf16  mean-relative (sum|err| / sum|ref|) <= 1e-2 and
        max-abs <= 3e-2 * max(1, max|ref|).  Beyond the forward's roundings the
        backward stores the walked queries X_b^(c), their gradients G and
        every output in bf16 (2^-9 relative each), and dS = P (dP - D) loses
        digits where dP is close to D, so the forward's 5e-3 / 2e-2 bar is
        doubled and the max-abs bar scaled to the gradient's size.
"""
import numpy as np
import pytest
import torch

import householder_softmax_attention_gb300 as pa
from oracle.chunked_bwd import path_chunked_bwd
from seeded_inputs import Workload, make_grad_inputs, make_inputs

pytestmark = pytest.mark.gpu

NAMES = ["dq", "dk", "dv", "dw", "dbeta", "dlogf"]


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _run(wl, with_dlse=True):
    x = make_inputs(wl)
    gi = make_grad_inputs(wl, with_dlse=with_dlse)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in {**x, **gi}.items()}
    out, lse = pa.path_attn_fwd(dev["q"], dev["k"], dev["v"], dev["w"], dev["beta"], dev["logf"],
                                scale=x["scale"])
    grads = pa.path_attn_bwd(dev["q"], dev["k"], dev["v"], dev["w"], dev["beta"], out, lse,
                             dev["dout"], logf=dev["logf"], scale=x["scale"], dlse=dev["dlse"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, clear=True) == 0
    return x, gi, out, lse, grads


def _oracle(x, gi, b, h):
    sel = lambda t: None if t is None else _np(t[b, h])
    return path_chunked_bwd(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["w"]), sel(x["beta"]),
                            sel(gi["dout"]), 16, logf=sel(x["logf"]), scale=x["scale"],
                            dlse=sel(gi["dlse"]))


def _compare(dtype, got, ref, name):
    err = np.abs(got - ref)
    big = max(1.0, float(np.abs(ref).max()))
    if float(np.abs(ref).max()) == 0.0:  # e.g. T = 1: one key, softmax constant
        assert err.max() <= (3e-2 if dtype == "bf16" else 1e-4), (name, err.max())
        return
    if dtype == "bf16":
        mrel = err.sum() / max(np.abs(ref).sum(), 1e-30)
        assert mrel <= 1e-2, (name, mrel)
        assert err.max() <= 3e-2 * big, (name, err.max(), big)
    else:
        assert err.max() <= 1e-4 * big, (name, err.max(), big)


@pytest.mark.parametrize("dtype,d,fox,T,dlse", [
    ("f32", 64, False, 150, True), ("f32", 64, True, 150, True), ("f32", 128, False, 130, False),
    ("bf16", 128, False, 300, True), ("bf16", 128, True, 300, True), ("bf16", 64, False, 200, False),
    ("bf16", 64, True, 260, True), ("bf16", 128, False, 40, True), ("f32", 64, False, 1, True),
    ("bf16", 128, False, 1, False)])
def test_backward_matches_oracle(dtype, d, fox, T, dlse):
    wl = Workload("bwd", 1, 2, T, d, dtype, fox=fox, seed=53)
    x, gi, _, _, grads = _run(wl, with_dlse=dlse)
    for h in range(2):
        ref = _oracle(x, gi, 0, h)
        for name, g, r in zip(NAMES, grads, ref):
            _compare(dtype, _np(g[0, h]), r, name)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_backward_near_reflections_matches_oracle(dtype, d):
    """beta near 2 keeps long paths alive (random beta damps distant logits)."""
    wl = Workload("bwd_refl", 1, 1, 400, d, dtype, beta_range=(1.95, 2.0), seed=54)
    x, gi, _, _, grads = _run(wl)
    ref = _oracle(x, gi, 0, 0)
    for name, g, r in zip(NAMES, grads, ref):
        _compare(dtype, _np(g[0, 0]), r, name)


def test_backward_multi_chunk_bf16_matches_oracle():
    wl = Workload("bwd_long", 1, 2, 1100, 128, "bf16", fox=True, seed=55)
    x, gi, _, _, grads = _run(wl)
    for h in range(2):
        ref = _oracle(x, gi, 0, h)
        for name, g, r in zip(NAMES, grads, ref):
            _compare("bf16", _np(g[0, h]), r, name)


@pytest.mark.parametrize("T,d,H,fox", [(4096, 128, 4, True), (16384, 128, 1, False)])
def test_backward_identities_at_size(T, d, H, fox):
    """Identities of the exact gradients, at sizes the oracle cannot finish:
    sum_j dv_j = sum_i dO_i (softmax rows sum to one); sum q.dq = sum k.dk
    (the PaTH logit is bilinear in q and k); sum v.dv = sum O.dO (O is linear
    in v); dlogf_0 = 0 (log f_0 enters every gate difference twice)."""
    wl = Workload("bwd_big", 1, H, T, d, "bf16", fox=fox, seed=56)
    x, gi, out, _, grads = _run(wl, with_dlse=False)
    dq, dk, dv, dw, dbeta, dlogf = (None if g is None else g.double() for g in grads)
    q, k, v = (x[n].cuda().double() for n in ("q", "k", "v"))
    dout = gi["dout"].cuda().double()
    o = out.double()
    rel = lambda a, b: float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))
    assert rel(dv.sum(dim=2), dout.sum(dim=2)) <= 2e-2
    qd = (q * dq).sum(dim=(2, 3))
    kd = (k * dk).sum(dim=(2, 3))
    scale_qd = (q * dq).abs().sum(dim=(2, 3))
    assert float(((qd - kd).abs() / scale_qd).max()) <= 1e-2
    vd = (v * dv).sum(dim=(2, 3))
    od = (o * dout).sum(dim=(2, 3))
    scale_vd = (v * dv).abs().sum(dim=(2, 3))
    assert float(((vd - od).abs() / scale_vd).max()) <= 1e-2
    if fox:
        assert float(dlogf[..., 0].abs().max()) <= 1e-2 * float(dlogf.abs().max())
    for g in (dq, dk, dv, dw, dbeta):
        assert bool(torch.isfinite(g).all())


@pytest.mark.parametrize("dtype,d,fox,T", [("f32", 64, True, 70), ("f32", 128, False, 40),
                                           ("bf16", 64, True, 100), ("bf16", 128, False, 64)])
def test_backward_matches_literal_autograd_oracle(dtype, d, fox, T):
    """The GPU gradients directly against autograd of the literal fp64
    forward (oracle/backward.py: every logit k_j^T H_{j+1} ... H_i q_i formed
    token by token), not only against the blockwise backward: one head,
    ragged against the chunk at T = 70 and 100."""
    from oracle.backward import path_oracle_bwd
    wl = Workload("bwd_literal", 1, 1, T, d, dtype, fox=fox, seed=57 + T)
    x, gi, _, _, grads = _run(wl, with_dlse=True)
    sel = lambda t: None if t is None else _np(t[0, 0])
    ref = path_oracle_bwd(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["w"]), sel(x["beta"]),
                          sel(gi["dout"]), logf=sel(x["logf"]), scale=x["scale"],
                          dlse=sel(gi["dlse"]))
    names = ["q", "k", "v", "w", "beta"] + (["logf"] if fox else [])
    for n, g in zip(names, grads):
        _compare(dtype, _np(g[0, 0]), ref[n].numpy(), "d" + n)
