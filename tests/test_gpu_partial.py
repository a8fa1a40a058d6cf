"""GPU parity of partial PaTH (PaTH on the first r head dimensions, no position
encoding on the rest; the authors' proposal in the OpenReview discussion,
sections "Efficiency" and "NoPE not included as a baseline") against the fp64
oracle's own partial-PaTH definition.  Tolerances as for the forward: fp32
1e-4 max-abs; bf16 2e-2 max-abs and 5e-3 mean-relative on out, 2e-2 on lse.
"""
import numpy as np
import pytest
import torch

import householder_softmax_attention_gb300 as pa
from oracle import path_oracle_partial_fwd
from seeded_inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _subspace_u(x, r, seed):
    """A unit u in R^r per token, drawn like w (the generator's w is in R^d)."""
    g = torch.Generator().manual_seed(seed)
    B, H, T, _ = x["q"].shape
    u = torch.randn((B, H, T, r), generator=g)
    u = u / u.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    return u.to(x["q"].dtype).contiguous()


@pytest.mark.parametrize("dtype,d,r,fox,T", [
    ("f32", 64, 0, False, 300), ("f32", 64, 16, True, 300), ("f32", 64, 64, False, 300),
    ("bf16", 128, 32, False, 300), ("bf16", 128, 64, True, 300), ("bf16", 64, 24, False, 300),
    ("bf16", 128, 64, False, 2048), ("bf16", 128, 64, False, 1000), ("bf16", 128, 64, True, 129),
    ("bf16", 128, 64, False, 1), ("bf16", 128, 0, False, 300), ("bf16", 128, 128, True, 300)])
def test_partial_path_matches_oracle(dtype, d, r, fox, T):
    wl = Workload("partial", 1, 2, T, d, dtype, fox=fox, seed=41)
    x = make_inputs(wl)
    u = _subspace_u(x, r, 42)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    out, lse = pa.path_attn_fwd_partial(dev["q"], dev["k"], dev["v"], u.cuda(), dev["beta"],
                                        dev["logf"], scale=x["scale"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, clear=True) == 0
    ref, ref_lse = path_oracle_partial_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), _np(u),
                                           _np(x["beta"]),
                                           None if x["logf"] is None else _np(x["logf"]),
                                           scale=x["scale"])
    got, got_lse = _np(out), _np(lse)
    err = np.abs(got - ref)
    if dtype == "bf16":
        assert err.max() <= 2e-2, err.max()
        assert err.sum() / np.abs(ref).sum() <= 5e-3
        assert np.abs(got_lse - ref_lse).max() <= 2e-2
    else:
        assert err.max() <= 1e-4, err.max()
        assert np.abs(got_lse - ref_lse).max() <= 1e-4


def _padded(u, d):
    """u [B, H, T, r] widened with zeros to d columns: full PaTH on the padded
    directions is partial PaTH on the first r coordinates."""
    B, H, T, r = u.shape
    w = torch.zeros((B, H, T, d), dtype=u.dtype, device=u.device)
    w[..., :r] = u
    return w


@pytest.mark.parametrize("fox", [False, True])
def test_rank64_kernel_matches_full_kernels_on_padded_directions(fox):
    """bf16, d = 128, r = 64 runs the rank-64 kernels (the attention carries
    64 coordinates through the transitions, the preparation reads u through a
    64-column tensor map); the full kernels on the zero-padded directions
    compute every product term identically, so the outputs agree bit for bit."""
    wl = Workload("partial_eq", 2, 3, 1100, 128, "bf16", fox=fox, seed=43)
    x = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in make_inputs(wl).items()}
    u = _subspace_u(x, 64, 44).cuda()
    o1, l1 = pa.path_attn_fwd_partial(x["q"], x["k"], x["v"], u, x["beta"], x["logf"],
                                      scale=x["scale"])
    o2, l2 = pa.path_attn_fwd(x["q"], x["k"], x["v"], _padded(u, 128), x["beta"], x["logf"],
                              scale=x["scale"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, clear=True) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("beta_range", [None, (1.98, 2.0)])
@pytest.mark.parametrize("fox", [False, True])
def test_rank64_full_length_sampled(fox, beta_range):
    """The headline shape (B=2, H=16, T=16384, d=128) with r = 64: sampled rows
    of four heads (row T-1 and the boundary rows of the first and last four
    chunks among them) against the oracle, run as full PaTH on the
    zero-padded directions (pinned equal to the partial definition)."""
    from oracle import path_oracle_fwd
    from seeded_inputs import WORKLOADS, sample_rows
    wl = WORKLOADS["t16k_d128"].with_(fox=fox, beta_range=beta_range, seed=47 + int(fox))
    x = make_inputs(wl, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(48)
    u = torch.randn((wl.B, wl.H, wl.T, 64), generator=g, device="cuda")
    u = (u / u.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(torch.bfloat16).contiguous()
    out, lse = pa.path_attn_fwd_partial(x["q"], x["k"], x["v"], u, x["beta"], x["logf"],
                                        scale=x["scale"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, clear=True) == 0
    heads = [(0, 0), (1, 15), (0, 9), (1, 4)]
    rows = sample_rows(wl.T, 128, 12, seed=49)
    sel = lambda t: None if t is None else torch.stack([t[b, h] for b, h in heads]).float().cpu().numpy()
    flat = [i * wl.T + r for i in range(len(heads)) for r in rows]
    ro, rl = path_oracle_fwd(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(_padded(u, 128)),
                             sel(x["beta"]), sel(x["logf"]), x["scale"], rows=flat)
    go = sel(out).reshape(-1, 128)[flat].astype(np.float64)
    gl = sel(lse).reshape(-1)[flat].astype(np.float64)
    err = np.abs(go - ro)
    print(f"PARTIAL r=64 fox={fox} beta={beta_range}: max_abs {err.max():.3e} "
          f"mean_rel {err.sum() / np.abs(ro).sum():.3e} lse {np.abs(gl - rl).max():.3e}")
    assert err.max() <= 2e-2
    assert err.sum() / np.abs(ro).sum() <= 5e-3
    assert np.abs(gl - rl).max() <= 2e-2
