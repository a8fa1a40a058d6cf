"""Seeded synthetic inputs for PaTH attention workloads.

This module is shared by the tests, the smoke check and the bench.  It holds
no arithmetic of the method: it only draws random tensors with the shapes and
distributions of the workloads and hands them out.  Both the CUDA path and the
CPU oracle consume what it returns; neither is imported here.

Recipe (every workload):
  q, k, v ~ N(0, 1);  w ~ N(0, 1) then L2-normalised per (token, head) in fp32;
  beta = 2 * sigmoid(N(0, 1)) in fp32;  scale = 1/sqrt(d);  causal.
Options:
  near_reflection -- a seeded 10% of tokens get beta ~ U[1.9, 2.0)
  fox             -- log f_t = log(sigmoid(N(2, 1))) in fp32 (PaTH-FoX gate)
  beta_range      -- draw every beta ~ U[lo, hi) instead (stress cases)
  w_spread        -- nearly equal directions: per (b, h) one unit vector u,
                     then w_t = u + w_spread * N(0, I) / sqrt(d), L2-normalised
                     (every Gram entry of a chunk close to 1; stress case)
The shapes follow the B x T x d grid of the PaTH authors' kernel-latency table
(OpenReview rebuttal, "Efficiency Evaluation"), with H = 16 heads at d = 128
and H = 32 at d = 64.  No dataset is involved.

The generator lives on ``device`` (CPU by default), so a given seed gives the
same values on every machine for CPU generation; device generation is faster
for the large workloads and is deterministic per device type.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dtype: str = "bf16"          # "bf16" or "f32"
    near_reflection: bool = False
    fox: bool = False
    beta_range: tuple | None = None
    w_spread: float | None = None
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads, named by what they are.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 2, 256, 64, "f32",
                         note="tiny PaTH forward in fp32; oracle runs in full"),
    "t2k_d128": Workload("t2k_d128", 16, 16, 2048, 128),
    "t2k_d64": Workload("t2k_d64", 16, 32, 2048, 64),
    "t4k_d128_refl": Workload("t4k_d128_refl", 8, 16, 4096, 128, near_reflection=True),
    "t4k_d64_refl": Workload("t4k_d64_refl", 8, 32, 4096, 64, near_reflection=True),
    "fox_t8k_d128": Workload("fox_t8k_d128", 4, 16, 8192, 128, fox=True),
    "t16k_d128": Workload("t16k_d128", 2, 16, 16384, 128,
                          note="long-context headline roofline workload"),
    "fox_t16k_d128": Workload("fox_t16k_d128", 2, 16, 16384, 128, fox=True,
                              note="the headline shape with the FoX gate"),
    "t16k_d64": Workload("t16k_d64", 2, 32, 16384, 64),
}


def make_inputs(wl: Workload, device="cpu"):
    """Draw the inputs of ``wl``.  Returns a dict with q, k, v, w ([B,H,T,d] in
    the workload dtype), beta ([B,H,T] fp32), logf ([B,H,T] fp32 or None) and
    scale (python float)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed)
    shape = (wl.B, wl.H, wl.T, wl.d)

    def normal(shp, mean=0.0):
        x = torch.randn(shp, generator=g, device=dev, dtype=torch.float32)
        return x + mean if mean else x

    q = normal(shape)
    k = normal(shape)
    v = normal(shape)
    w = normal(shape)
    w = w / w.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    if wl.w_spread is not None:
        u = normal((wl.B, wl.H, 1, wl.d))
        u = u / u.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        w = u + (wl.w_spread / math.sqrt(wl.d)) * normal(shape)
        w = w / w.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    bshape = shape[:-1]
    if wl.beta_range is not None:
        lo, hi = wl.beta_range
        beta = lo + (hi - lo) * torch.rand(bshape, generator=g, device=dev)
    else:
        beta = 2.0 * torch.sigmoid(normal(bshape))
    if wl.near_reflection:
        pick = torch.rand(bshape, generator=g, device=dev) < 0.10
        hi_beta = 1.9 + 0.1 * torch.rand(bshape, generator=g, device=dev)
        beta = torch.where(pick, hi_beta, beta)
    beta = beta.clamp(0.0, 2.0).contiguous()
    logf = None
    if wl.fox:
        logf = torch.log(torch.sigmoid(normal(bshape, 2.0))).contiguous()
    dt = wl.torch_dtype
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(),
                v=v.to(dt).contiguous(), w=w.to(dt).contiguous(),
                beta=beta, logf=logf, scale=1.0 / math.sqrt(wl.d))


def make_grad_inputs(wl: Workload, device="cpu", with_dlse=True):
    """Upstream gradients for the backward of ``wl``'s forward: dout
    ([B,H,T,d], workload dtype) ~ N(0, 1) and dlse ([B,H,T] fp32) ~ N(0, 1)
    (None without ``with_dlse``), from their own seed."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed + 7919)
    shape = (wl.B, wl.H, wl.T, wl.d)
    dout = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    dlse = torch.randn(shape[:-1], generator=g, device=dev, dtype=torch.float32)
    return dict(dout=dout.to(wl.torch_dtype).contiguous(),
                dlse=dlse.contiguous() if with_dlse else None)


# Decoding: one new token per (b, h) against a cache of Tmax rows.
DECODE_WORKLOADS = {
    "decode_t16k_d128": Workload("decode_t16k_d128", 2, 16, 16384, 128,
                                 note="one decoding step at position T - 1 of a 16K cache"),
    "decode_t16k_d64": Workload("decode_t16k_d64", 2, 32, 16384, 64),
}


def make_decode_inputs(wl: Workload, device="cpu"):
    """Draw one decoding step of ``wl`` (T = cache rows): the new token's q, k,
    v, w ([B,H,d], workload dtype), beta and logf ([B,H] fp32; logf only with
    ``wl.fox``), and a synthetic cache state: kcache ~ N(0, 1) fp32 and vcache
    ~ N(0, 1) ([B,H,T,d]); with ``wl.fox`` a decreasing lamcache ([B,H,T] fp32,
    steps ~ U[0, 0.1)).  Returns a dict (also ``scale``)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed + 104729)
    B, H, T, d = wl.B, wl.H, wl.T, wl.d
    dt = wl.torch_dtype

    def normal(shp):
        return torch.randn(shp, generator=g, device=dev, dtype=torch.float32)

    q, k, v, w = (normal((B, H, d)) for _ in range(4))
    w = w / w.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    beta = (2.0 * torch.sigmoid(normal((B, H)))).clamp(0.0, 2.0).contiguous()
    kcache = normal((B, H, T, d)).contiguous()
    vcache = normal((B, H, T, d)).to(dt).contiguous()
    logf = lamcache = None
    if wl.fox:
        logf = torch.log(torch.sigmoid(normal((B, H)) + 2.0)).contiguous()
        steps = 0.1 * torch.rand((B, H, T), generator=g, device=dev)
        lamcache = (-torch.cumsum(steps, dim=-1)).contiguous()
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                w=w.to(dt).contiguous(), beta=beta, logf=logf, kcache=kcache, vcache=vcache,
                lamcache=lamcache, scale=1.0 / math.sqrt(d))


# The w / beta producer: hidden states x [B, T, Dm] with Dm = H * d, a rank-R
# projection (R not on the pages: 64).
@dataclass(frozen=True)
class ProducerWorkload:
    name: str
    B: int
    T: int
    Dm: int
    H: int
    d: int
    R: int
    dtype: str = "bf16"
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


PRODUCER_WORKLOADS = {
    "producer_t16k_d128": ProducerWorkload("producer_t16k_d128", 2, 16384, 2048, 16, 128, 64),
    "producer_t16k_d64": ProducerWorkload("producer_t16k_d64", 2, 16384, 2048, 32, 64, 64),
}


def make_producer_inputs(wl: ProducerWorkload, device="cpu"):
    """x ~ N(0, 1); Wd ~ N(0, 1/Dm); Wu ~ N(0, 1/R); conv taps ~ N(0, 1/3);
    Ub ~ N(0, 1/Dm); bb ~ N(0, 1).  x and the matrices in the workload dtype,
    taps and bias fp32."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed + 7)
    dt = wl.torch_dtype

    def normal(shp, std):
        return std * torch.randn(shp, generator=g, device=dev, dtype=torch.float32)

    x = normal((wl.B, wl.T, wl.Dm), 1.0)
    Wd = normal((wl.R, wl.Dm), wl.Dm ** -0.5)
    Wu = normal((wl.H * wl.d, wl.R), wl.R ** -0.5)
    cw = normal((wl.H * wl.d, 3), 3 ** -0.5)
    Ub = normal((wl.H, wl.Dm), wl.Dm ** -0.5)
    bb = normal((wl.H,), 1.0)
    return dict(x=x.to(dt).contiguous(), Wd=Wd.to(dt).contiguous(), Wu=Wu.to(dt).contiguous(),
                cw=cw.contiguous(), Ub=Ub.to(dt).contiguous(), bb=bb.contiguous())


def sample_rows(T: int, C: int, n_extra: int, seed: int = 0):
    """A fixed, seeded set of query rows of one head for sampled parity checks:
    the first and last rows, chunk boundaries around the first and last four
    chunks, and ``n_extra`` random rows.  Returned sorted and unique."""
    g = torch.Generator().manual_seed(seed + 7919)
    rows = {0, T - 1}
    n = -(-T // C)
    for c in list(range(min(4, n))) + list(range(max(0, n - 4), n)):
        for r in (c * C - 1, c * C, c * C + 1, c * C + C - 1):
            if 0 <= r < T:
                rows.add(r)
    if n_extra > 0:
        rows.update(torch.randint(0, T, (n_extra,), generator=g).tolist())
    return sorted(rows)
