"""Pins for the gradient oracle (``oracle/backward.py``): its forward equals the
pinned C oracle, its gradients equal central finite differences of that
forward for every input, and with beta = 0 they equal the gradients of plain
causal attention (torch's scaled_dot_product_attention, fp64).
"""
import numpy as np
import pytest
import torch

from oracle import path_oracle_fwd
from oracle.backward import path_attn_literal, path_oracle_bwd


def _inputs(seed, T, d, fox):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)
    q, k, v, w = r(T, d), r(T, d), r(T, d), r(T, d)
    w = w / w.norm(dim=-1, keepdim=True)
    beta = 2 * torch.sigmoid(r(T))
    logf = torch.log(torch.sigmoid(r(T) + 2)) if fox else None
    return q, k, v, w, beta, logf


@pytest.mark.parametrize("fox", [False, True])
def test_literal_forward_is_the_c_oracle(fox):
    q, k, v, w, beta, logf = _inputs(61, 13, 5, fox)
    out, lse = path_attn_literal(q, k, v, w, beta, logf, scale=0.45)
    ref_out, ref_lse = path_oracle_fwd(q.numpy(), k.numpy(), v.numpy(), w.numpy(), beta.numpy(),
                                       None if logf is None else logf.numpy(), scale=0.45)
    np.testing.assert_allclose(out.numpy(), ref_out, atol=1e-12)
    np.testing.assert_allclose(lse.numpy(), ref_lse, atol=1e-12)


@pytest.mark.parametrize("fox", [False, True])
def test_gradients_match_central_differences(fox):
    T, d, scale = 7, 4, 0.6
    q, k, v, w, beta, logf = _inputs(62, T, d, fox)
    g = torch.Generator().manual_seed(63)
    dout = torch.randn(T, d, generator=g, dtype=torch.float64)
    dlse = torch.randn(T, generator=g, dtype=torch.float64)
    grads = path_oracle_bwd(q, k, v, w, beta, dout, logf, scale, dlse)
    inputs = {"q": q, "k": k, "v": v, "w": w, "beta": beta}
    if fox:
        inputs["logf"] = logf

    def loss(vals):
        out, lse = path_attn_literal(vals["q"], vals["k"], vals["v"], vals["w"], vals["beta"],
                                     vals.get("logf"), scale)
        return float((out * dout).sum() + (lse * dlse).sum())

    eps = 1e-6
    for name, x in inputs.items():
        fd = torch.zeros_like(x)
        flat = x.reshape(-1)
        for n in range(flat.numel()):
            plus = {m: t.clone() for m, t in inputs.items()}
            minus = {m: t.clone() for m, t in inputs.items()}
            plus[name].reshape(-1)[n] += eps
            minus[name].reshape(-1)[n] -= eps
            fd.reshape(-1)[n] = (loss(plus) - loss(minus)) / (2 * eps)
        np.testing.assert_allclose(grads[name].numpy(), fd.numpy(), atol=1e-7, rtol=1e-6,
                                   err_msg=name)


def test_beta_zero_gradients_are_plain_attention_gradients():
    T, d, scale = 11, 6, 0.4
    q, k, v, w, beta, _ = _inputs(64, T, d, False)
    beta = torch.zeros(T, dtype=torch.float64)
    g = torch.Generator().manual_seed(65)
    dout = torch.randn(T, d, generator=g, dtype=torch.float64)
    grads = path_oracle_bwd(q, k, v, w, beta, dout, scale=scale)
    qs, ks, vs = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qs[None, None], ks[None, None],
                                                         vs[None, None], is_causal=True,
                                                         scale=scale)[0, 0]
    ref = torch.autograd.grad((o * dout).sum(), [qs, ks, vs])
    for name, r in zip("qkv", ref):
        np.testing.assert_allclose(grads[name].numpy(), r.numpy(), atol=1e-12, err_msg=name)
    # with beta = 0 the transitions do not depend on w
    assert float(grads["w"].abs().max()) == 0.0
