"""Gradient oracle for PaTH / PaTH-FoX attention -- TEST INFRASTRUCTURE.

Only ``tests/`` may import this module.

The pages define the forward only ("PaTH Attention: Position Encoding via
Accumulating Householder Transformations", slides, frames "PaTH inserts a
learned transformation along every path" and "FoX adds a separate mechanism
for forgetting"; the OpenReview discussion times the forward and backward
together, section "Efficiency Evaluation").  The gradient is therefore that of
the forward's definition: the forward below is written literally in fp64
PyTorch CPU ops (H_t as explicit d x d matrices, each logit
k_j^T H_{j+1} ... H_i q_i formed by walking from H_i down to H_{j+1}), and
torch.autograd differentiates it.  Cost O(T^2 d^2) with a Python loop over
rows: small problems only.
"""
from __future__ import annotations

import torch


def path_attn_literal(q, k, v, w, beta, logf=None, scale=None):
    """Literal PaTH(-FoX) forward of one head in fp64 torch (differentiable).
    q, k, v, w: [T, d]; beta, logf: [T].  Returns (out [T, d], lse [T])."""
    T, d = q.shape
    if scale is None:
        scale = d ** -0.5
    eye = torch.eye(d, dtype=q.dtype)
    H = [eye - beta[t] * torch.outer(w[t], w[t]) for t in range(T)]
    gate = torch.cumsum(logf, 0) if logf is not None else None
    outs, lses = [], []
    for i in range(T):
        z = q[i]
        logits = [None] * (i + 1)
        for j in range(i, -1, -1):
            logits[j] = scale * (k[j] @ z)          # z = H_{j+1} ... H_i q_i
            if gate is not None:
                logits[j] = logits[j] + (gate[i] - gate[j])
            z = H[j] @ z                            # cross token j
        s = torch.stack(logits)
        lse = torch.logsumexp(s, 0)
        outs.append(torch.softmax(s, 0) @ v[: i + 1])
        lses.append(lse)
    return torch.stack(outs), torch.stack(lses)


def path_oracle_bwd(q, k, v, w, beta, dout, logf=None, scale=None, dlse=None):
    """Gradients of sum(out * dout) (+ sum(lse * dlse)) with respect to
    q, k, v, w, beta (and logf) for one head, in fp64.  Returns a dict."""
    names = ["q", "k", "v", "w", "beta"] + (["logf"] if logf is not None else [])
    xs = {n: torch.as_tensor(a, dtype=torch.float64).clone().requires_grad_(True)
          for n, a in zip(names, [q, k, v, w, beta] + ([logf] if logf is not None else []))}
    out, lse = path_attn_literal(xs["q"], xs["k"], xs["v"], xs["w"], xs["beta"], xs.get("logf"),
                                 scale)
    loss = (out * torch.as_tensor(dout, dtype=torch.float64)).sum()
    if dlse is not None:
        loss = loss + (lse * torch.as_tensor(dlse, dtype=torch.float64)).sum()
    grads = torch.autograd.grad(loss, [xs[n] for n in names])
    return {n: g.detach() for n, g in zip(names, grads)}
