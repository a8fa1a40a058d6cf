"""The blockwise backward (``oracle/chunked_bwd.py``, the blueprint of a GPU
backward) against the autograd gradient oracle, which is itself pinned to
finite differences (``tests/test_backward_oracle.py``)."""
import numpy as np
import pytest
import torch

from oracle.backward import path_oracle_bwd
from oracle.chunked_bwd import path_chunked_bwd


@pytest.mark.parametrize("T,d,C,fox,refl", [(45, 8, 8, False, False), (45, 8, 8, True, False),
                                            (32, 6, 16, False, True), (29, 5, 4, True, True),
                                            (7, 4, 8, False, False)])
def test_blockwise_backward_matches_autograd(T, d, C, fox, refl):
    g = np.random.default_rng(71 + T + C)
    q, k, v, w = (g.standard_normal((T, d)) for _ in range(4))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = 2.0 / (1.0 + np.exp(-g.standard_normal(T)))
    if refl:
        beta[g.random(T) < 0.3] = 1.97
    logf = np.log(1.0 / (1.0 + np.exp(-(g.standard_normal(T) + 2.0)))) if fox else None
    dout = g.standard_normal((T, d))
    scale = 0.55
    got = path_chunked_bwd(q, k, v, w, beta, dout, C, logf=logf, scale=scale)
    ref = path_oracle_bwd(*(torch.from_numpy(x) for x in (q, k, v, w, beta, dout)),
                          logf=None if logf is None else torch.from_numpy(logf), scale=scale)
    names = ["q", "k", "v", "w", "beta"] + (["logf"] if fox else [])
    for name, gv in zip(names, got):
        np.testing.assert_allclose(gv, ref[name].numpy(), atol=1e-9, rtol=1e-8, err_msg=name)


@pytest.mark.parametrize("fox", [False, True])
def test_blockwise_backward_with_lse_gradient_matches_autograd(fox):
    T, d, C, scale = 37, 6, 8, 0.5
    g = np.random.default_rng(83)
    q, k, v, w = (g.standard_normal((T, d)) for _ in range(4))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = 2.0 / (1.0 + np.exp(-g.standard_normal(T)))
    logf = np.log(1.0 / (1.0 + np.exp(-(g.standard_normal(T) + 2.0)))) if fox else None
    dout, dlse = g.standard_normal((T, d)), g.standard_normal(T)
    got = path_chunked_bwd(q, k, v, w, beta, dout, C, logf=logf, scale=scale, dlse=dlse)
    ref = path_oracle_bwd(*(torch.from_numpy(x) for x in (q, k, v, w, beta, dout)),
                          logf=None if logf is None else torch.from_numpy(logf), scale=scale,
                          dlse=torch.from_numpy(dlse))
    names = ["q", "k", "v", "w", "beta"] + (["logf"] if fox else [])
    for name, gv in zip(names, got):
        np.testing.assert_allclose(gv, ref[name].numpy(), atol=1e-9, rtol=1e-8, err_msg=name)
