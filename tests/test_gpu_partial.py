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
    ("bf16", 128, 64, False, 2048)])
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
