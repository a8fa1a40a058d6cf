"""PaTH attention forward pass on one GB300 (sm_103a).

A thin ctypes binding of ``libpathattn.so`` (C ABI in ``include/pathattn.h``).
It only marshals arguments: every step of the forward pass runs in the
library's CUDA kernels.  torch is used for device memory and the current
stream.  If the library is missing, every call raises; there is no fallback.

The operation ("PaTH Attention: Position Encoding via Accumulating Householder
Transformations", discussion slides, frames "PaTH inserts a learned
transformation along every path" and "FoX adds a separate mechanism for
forgetting"):

    s_ij = scale * k_j^T H_{j+1} ... H_i q_i [+ sum_{s=j+1}^{i} log f_s],
    H_t = I - beta_t w_t w_t^T,   o_i = sum_{j<=i} softmax_j(s_ij) v_j.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "PathAttnError", "load_library", "path_attn_fwd", "path_attn_fwd_host",
    "path_attn_fwd_noalloc", "path_attn_noalloc_status", "path_attn_debug_wait_timeout",
    "path_attn_prefill",
    "path_attn_decode_step", "DecodeCache", "path_attn_fwd_partial", "path_producer_fwd",
    "path_attn_bwd", "path_attn_bwd_workspace_bytes", "path_attn_bwd_launches_per_call",
    "path_attn_debug_factors", "path_attn_device_status", "path_attn_workspace_bytes",
    "path_attn_chunk_size", "path_attn_launches_per_call", "path_attn_set_transition_form",
    "path_attn_timing_enable",
    "path_attn_timing_read", "path_attn_bwd_timing_read", "BWD_PHASES", "path_attn_version",
    "path_attn_status_string",
    "LIBRARY_PATH", "HEADER_PATH", "PATH_DTYPE_F32", "PATH_DTYPE_BF16",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libpathattn.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "pathattn.h")

PATH_OK = 0
PATH_DTYPE_F32 = 0
PATH_DTYPE_BF16 = 1

_lock = threading.Lock()
_lib = None


class PathAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if _lib is not None:
            name = _lib.path_attn_status_string(status).decode()
            last = _lib.path_attn_last_error().decode()
            detail = f"{name}" + (f" ({last})" if last else "")
        super().__init__(f"{what} failed: status {status} {detail}")


def load_library(path: str | None = None):
    """Load libpathattn.so (built by ``build.py``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIBRARY_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libpathattn.so not found at {p}; build it with "
                "`python -m householder_softmax_attention_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, fp, i, f = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fwd_args = [vp, vp, vp, vp, fp, fp, f, vp, fp, i, i, i, i, i, vp]
        lib.path_attn_fwd.argtypes = fwd_args
        lib.path_attn_fwd.restype = i
        lib.path_attn_fwd_host.argtypes = fwd_args
        lib.path_attn_fwd_host.restype = i
        lib.path_attn_status_string.argtypes = [i]
        lib.path_attn_status_string.restype = ctypes.c_char_p
        lib.path_attn_last_error.argtypes = []
        lib.path_attn_last_error.restype = ctypes.c_char_p
        lib.path_attn_version.argtypes = []
        lib.path_attn_version.restype = i
        lib.path_attn_workspace_bytes.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.path_attn_workspace_bytes.restype = i
        lib.path_attn_chunk_size.argtypes = [i, i]
        lib.path_attn_chunk_size.restype = i
        lib.path_attn_device_status.argtypes = [i, i]
        lib.path_attn_device_status.restype = i
        lib.path_attn_timing_enable.argtypes = [i]
        lib.path_attn_timing_enable.restype = i
        lib.path_attn_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                              ctypes.POINTER(ctypes.c_double),
                                              ctypes.POINTER(ctypes.c_long)]
        lib.path_attn_timing_read.restype = i
        lib.path_attn_bwd_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ctypes.c_long)]
        lib.path_attn_bwd_timing_read.restype = i
        lib.path_attn_set_transition_form.argtypes = [i]
        lib.path_attn_set_transition_form.restype = i
        lib.path_attn_launches_per_call.argtypes = [i, i, i]
        lib.path_attn_launches_per_call.restype = i
        lib.path_attn_bwd_launches_per_call.argtypes = [i, i, i, i]
        lib.path_attn_bwd_launches_per_call.restype = i
        lib.path_attn_debug_factors.argtypes = [vp, vp, vp, fp, fp, f, i, i, i, i, i,
                                                vp, vp, vp, vp, vp, vp]
        lib.path_attn_debug_factors.restype = i
        lib.path_attn_debug_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
        lib.path_attn_debug_wait_timeout.restype = i
        lib.path_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, fp, fp, f, vp, fp, vp,
                                              i, i, i, i, i, vp]
        lib.path_attn_fwd_noalloc.restype = i
        lib.path_attn_noalloc_status.argtypes = [i, i]
        lib.path_attn_noalloc_status.restype = i
        lib.path_attn_fwd_partial.argtypes = [vp, vp, vp, vp, fp, fp, f, vp, fp, i, i, i, i, i,
                                              i, vp]
        lib.path_attn_fwd_partial.restype = i
        lib.path_producer_fwd.argtypes = [vp, vp, vp, fp, vp, fp, vp, fp, i, i, i, i, i, i, i,
                                          vp]
        lib.path_producer_fwd.restype = i
        lib.path_attn_prefill.argtypes = [vp, vp, vp, vp, fp, fp, f, vp, fp, fp, vp, fp, i,
                                          i, i, i, i, i, vp]
        lib.path_attn_prefill.restype = i
        lib.path_attn_decode_step.argtypes = [vp, vp, vp, vp, fp, fp, f, fp, vp, fp, vp, i,
                                              vp, fp, i, i, i, i, i, vp]
        lib.path_attn_decode_step.restype = i
        lib.path_attn_bwd.argtypes = [vp, vp, vp, vp, fp, fp, f, vp, fp, vp, fp, vp, vp, vp, vp,
                                      fp, fp, i, i, i, i, i, vp]
        lib.path_attn_bwd.restype = i
        lib.path_attn_bwd_workspace_bytes.argtypes = [i, i, i, i, i, i,
                                                      ctypes.POINTER(ctypes.c_size_t)]
        lib.path_attn_bwd_workspace_bytes.restype = i
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != PATH_OK:
        raise PathAttnError(rc, what)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return PATH_DTYPE_BF16
    if t.dtype == torch.float32:
        return PATH_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_inputs(q, k, v, w, beta, logf, device_expected: bool):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("w", w)):
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, T, d]")
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    for name, t in (("beta", beta), ("logf", logf)):
        if t is None:
            continue
        if t.shape != q.shape[:-1] or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 [B, H, T] tensor")
    for t in (q, k, v, w, beta, logf):
        if t is not None and t.is_cuda != device_expected:
            raise ValueError("all tensors must be on " + ("the GPU" if device_expected else "the host"))
    if device_expected:
        dev = q.device
        for t in (k, v, w, beta, logf):
            if t is not None and t.device != dev:
                raise ValueError("all tensors must be on one device")


def path_attn_fwd(q, k, v, w, beta, logf=None, scale=None, out=None, lse=None,
                  want_lse=True, stream=None):
    """PaTH(-FoX) forward on CUDA tensors.

    q, k, v, w: ``[B, H, T, d]`` bfloat16 or float32 (one dtype), contiguous;
    beta (and logf for PaTH-FoX): ``[B, H, T]`` float32.  ``scale`` defaults to
    ``1/sqrt(d)``.  Returns ``(out, lse)`` (lse is None if ``want_lse`` is
    false).  Runs on ``stream`` (default: torch's current stream).
    """
    import torch
    lib = load_library()
    _check_inputs(q, k, v, w, beta, logf, True)
    B, H, T, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    st = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = lib.path_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(logf),
                               float(scale), _ptr(out), _ptr(lse), B, H, T, d,
                               _dtype_code(q), ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_attn_fwd")
    return out, lse


def path_attn_fwd_host(q, k, v, w, beta, logf=None, scale=None, out=None, lse=None,
                       want_lse=True, stream=None):
    """The same forward on host (CPU) tensors; copies to and from the current
    device happen inside the library call, which returns when the results are
    on the host.  Pinned host tensors make the copies faster."""
    import torch
    lib = load_library()
    _check_inputs(q, k, v, w, beta, logf, False)
    B, H, T, d = q.shape
    if scale is None:
        scale = d ** -0.5
    pin = q.is_pinned()  # outputs page-locked like the inputs, so copies overlap
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, pin_memory=pin)
    st = stream if stream is not None else torch.cuda.current_stream()
    rc = lib.path_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(logf),
                                float(scale), _ptr(out), _ptr(lse), B, H, T, d,
                                _dtype_code(q), ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_attn_fwd_host")
    return out, lse


def path_attn_fwd_noalloc(q, k, v, w, beta, logf=None, scale=None, out=None, lse=None,
                          status=None, want_lse=True, stream=None):
    """The forward through the allocation-free C entry, whose workspace is a
    static 64 MiB device array inside the library (for callers that may not
    allocate device memory).  Arguments as ``path_attn_fwd``; ``status`` is an
    optional device int32 tensor that receives the kernels' wait status.
    Output tensors are allocated here only when not passed in."""
    import torch
    lib = load_library()
    _check_inputs(q, k, v, w, beta, logf, True)
    B, H, T, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    st = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = lib.path_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(logf),
                                       float(scale), _ptr(out), _ptr(lse), _ptr(status),
                                       B, H, T, d, _dtype_code(q), ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_attn_fwd_noalloc")
    return out, lse


def path_attn_noalloc_status(device: int = 0, clear: bool = True) -> int:
    """0 if no bounded wait of ``path_attn_fwd_noalloc``'s kernels expired
    while they reported into the library's static status word (calls made
    with ``status=None``), else PATH_ERR_TIMEOUT.  Synchronises the device;
    allocates nothing."""
    return load_library().path_attn_noalloc_status(device, 1 if clear else 0)


def path_attn_fwd_partial(q, k, v, u, beta, logf=None, scale=None, out=None, lse=None,
                          want_lse=True, stream=None):
    """Partial PaTH on CUDA tensors: PaTH with ``u [B, H, T, r]`` on the first
    ``r`` head dimensions, no position encoding on the other ``d - r``.  Other
    arguments as ``path_attn_fwd``."""
    import torch
    lib = load_library()
    _check_inputs(q, k, v, q, beta, logf, True)
    B, H, T, d = q.shape
    if (u.dim() != 4 or u.shape[:3] != q.shape[:3] or u.dtype != q.dtype or not u.is_contiguous()
            or u.device != q.device or u.shape[3] > d):
        raise ValueError("u must be a contiguous [B, H, T, r] tensor like q, with r <= d")
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    st = stream if stream is not None else torch.cuda.current_stream(q.device)
    r = u.shape[3]
    with torch.cuda.device(q.device):
        rc = lib.path_attn_fwd_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(u) if r > 0 else None,
                                       _ptr(beta), _ptr(logf), float(scale), _ptr(out), _ptr(lse),
                                       B, H, T, d, r, _dtype_code(q), ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_attn_fwd_partial")
    return out, lse


def path_attn_bwd(q, k, v, w, beta, out, lse, dout, logf=None, scale=None, dlse=None,
                  grads=None, stream=None):
    """Gradients of a ``path_attn_fwd`` call on CUDA tensors.

    ``out`` and ``lse`` are the forward's results; ``dout [B, H, T, d]`` (q's
    dtype) and ``dlse [B, H, T]`` (float32, optional) are the gradients of the
    loss with respect to them.  Returns ``(dq, dk, dv, dw, dbeta, dlogf)``;
    dlogf is None without a gate.  ``grads`` may supply that tuple of output
    tensors to be written in place."""
    import torch
    lib = load_library()
    _check_inputs(q, k, v, w, beta, logf, True)
    B, H, T, d = q.shape
    for name, t, shape, dt in (("out", out, q.shape, q.dtype), ("dout", dout, q.shape, q.dtype),
                               ("lse", lse, q.shape[:-1], torch.float32),
                               ("dlse", dlse, q.shape[:-1], torch.float32)):
        if t is None and name == "dlse":
            continue
        if (t is None or t.shape != shape or t.dtype != dt or not t.is_contiguous()
                or t.device != q.device):
            raise ValueError(f"{name} must be a contiguous {dt} {tuple(shape)} tensor on q's device")
    if scale is None:
        scale = d ** -0.5
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(w),
                 torch.empty_like(beta), torch.empty_like(logf) if logf is not None else None)
    dq, dk, dv, dw, dbeta, dlogf = grads
    st = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = lib.path_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(logf),
                               float(scale), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dlse),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dw), _ptr(dbeta), _ptr(dlogf),
                               B, H, T, d, _dtype_code(q), ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_attn_bwd")
    return dq, dk, dv, dw, dbeta, dlogf


def path_attn_bwd_launches_per_call(T, d, dtype_code, with_gate=False) -> int:
    n = load_library().path_attn_bwd_launches_per_call(T, d, dtype_code, int(with_gate))
    if n < 0:
        raise PathAttnError(n, "path_attn_bwd_launches_per_call")
    return n


def path_attn_bwd_workspace_bytes(B, H, T, d, dtype_code, with_gate=False) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().path_attn_bwd_workspace_bytes(B, H, T, d, dtype_code, int(with_gate),
                                                        ctypes.byref(n)),
           "path_attn_bwd_workspace_bytes")
    return n.value


def path_producer_fwd(x, Wd, Wu, cw, Ub, bb, H, d, w=None, beta=None, stream=None):
    """w and beta from hidden states ``x [B, T, Dm]`` (bfloat16 or float32):
    low-rank projection ``Wd [R, Dm]``, ``Wu [H*d, R]``, causal width-3
    convolution ``cw [H*d, 3]`` (float32), per-head L2 normalization, and
    ``beta = 2 sigmoid(x Ub^T + bb)`` with ``Ub [H, Dm]``, ``bb [H]`` (float32).
    Returns ``(w [B, H, T, d], beta [B, H, T])``."""
    import torch
    lib = load_library()
    if x.dim() != 3 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA [B, T, Dm] tensor")
    B, T, Dm = x.shape
    R = Wd.shape[0]
    shapes = {"Wd": (Wd, (R, Dm), x.dtype), "Wu": (Wu, (H * d, R), x.dtype),
              "cw": (cw, (H * d, 3), torch.float32), "Ub": (Ub, (H, Dm), x.dtype),
              "bb": (bb, (H,), torch.float32)}
    for name, (t, shp, dt) in shapes.items():
        if tuple(t.shape) != shp or t.dtype != dt or not t.is_contiguous() or t.device != x.device:
            raise ValueError(f"{name} must be a contiguous {dt} tensor of shape {shp} on x's device")
    if w is None:
        w = torch.empty((B, H, T, d), device=x.device, dtype=x.dtype)
    if beta is None:
        beta = torch.empty((B, H, T), device=x.device, dtype=torch.float32)
    st = stream if stream is not None else torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        rc = lib.path_producer_fwd(_ptr(x), _ptr(Wd), _ptr(Wu), _ptr(cw), _ptr(Ub), _ptr(bb),
                                   _ptr(w), _ptr(beta), B, T, Dm, H, d, R, _dtype_code(x),
                                   ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_producer_fwd")
    return w, beta


class DecodeCache:
    """Device caches of one decoder (layout of ``include/pathattn.h``):
    ``kcache [B, H, Tmax, d]`` float32 (keys carried to the latest token),
    ``vcache [B, H, Tmax, d]`` in the model dtype, ``lamcache [B, H, Tmax]``
    float32 (gate prefixes; None without a gate)."""

    def __init__(self, B, H, Tmax, d, dtype, device, gated=False):
        import torch
        self.B, self.H, self.Tmax, self.d = B, H, Tmax, d
        self.kcache = torch.zeros((B, H, Tmax, d), device=device, dtype=torch.float32)
        self.vcache = torch.zeros((B, H, Tmax, d), device=device, dtype=dtype)
        self.lamcache = (torch.zeros((B, H, Tmax), device=device, dtype=torch.float32)
                         if gated else None)

    @classmethod
    def wrap(cls, kcache, vcache, lamcache=None):
        """A cache over existing tensors (kept, not copied)."""
        self = cls.__new__(cls)
        self.B, self.H, self.Tmax, self.d = kcache.shape
        import torch
        if kcache.dtype != torch.float32 or vcache.shape != kcache.shape:
            raise ValueError("kcache must be float32 and share [B, H, Tmax, d] with vcache")
        for t in (kcache, vcache, lamcache):
            if t is not None and not t.is_contiguous():
                raise ValueError("cache tensors must be contiguous")
        if lamcache is not None and lamcache.shape != kcache.shape[:-1]:
            raise ValueError("lamcache must be [B, H, Tmax]")
        self.kcache, self.vcache, self.lamcache = kcache, vcache, lamcache
        return self

    def rows(self, b0, b1):
        """The caches of batch rows b0..b1-1 (views of the same memory)."""
        return DecodeCache.wrap(self.kcache[b0:b1], self.vcache[b0:b1],
                                None if self.lamcache is None else self.lamcache[b0:b1])


def path_attn_prefill(q, k, v, w, beta, logf, cache: DecodeCache, scale=None, out=None,
                      lse=None, want_lse=True, stream=None):
    """``path_attn_fwd`` over a prompt that also fills rows ``0..T-1`` of
    ``cache`` (keys carried to the prompt end, values, gate prefixes)."""
    import torch
    lib = load_library()
    _check_inputs(q, k, v, w, beta, logf, True)
    B, H, T, d = q.shape
    if (B, H, d) != (cache.B, cache.H, cache.d) or cache.vcache.dtype != q.dtype:
        raise ValueError("cache does not match the inputs")
    if (logf is None) != (cache.lamcache is None):
        raise ValueError("a gated prompt needs a gated cache and the reverse")
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    st = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = lib.path_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(logf),
                                   float(scale), _ptr(out), _ptr(lse), _ptr(cache.kcache),
                                   _ptr(cache.vcache), _ptr(cache.lamcache), cache.Tmax,
                                   B, H, T, d, _dtype_code(q), ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_attn_prefill")
    return out, lse


def path_attn_decode_step(q, k, v, w, beta, logf, cache: DecodeCache, pos, max_len,
                          scale=None, out=None, lse=None, want_lse=True, stream=None):
    """One decoding step: ``q, k, v, w [B, H, d]``, ``beta`` (and ``logf``)
    ``[B, H]`` float32, ``pos`` a device int32 ``[B]`` tensor with each batch
    row's position, ``max_len`` a host bound above every ``pos[b]``.  Rewrites
    the cached keys in place, appends the new token, returns ``(out, lse)``."""
    import torch
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v), ("w", w)):
        if t.dim() != 3 or t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, d] tensor like q")
    B, H, d = q.shape
    for name, t in (("beta", beta), ("logf", logf)):
        if t is not None and (t.shape != (B, H) or t.dtype != torch.float32
                              or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 [B, H] tensor")
    if pos.dtype != torch.int32 or pos.shape != (B,) or not pos.is_cuda:
        raise ValueError("pos must be a device int32 [B] tensor")
    if (B, H, d) != (cache.B, cache.H, cache.d) or cache.vcache.dtype != q.dtype:
        raise ValueError("cache does not match the inputs")
    if (logf is None) != (cache.lamcache is None):
        raise ValueError("a gated step needs a gated cache and the reverse")
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H), device=q.device, dtype=torch.float32)
    st = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = lib.path_attn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(logf),
                                       float(scale), _ptr(cache.kcache), _ptr(cache.vcache),
                                       _ptr(cache.lamcache), _ptr(pos), int(max_len), _ptr(out),
                                       _ptr(lse), B, H, cache.Tmax, d, _dtype_code(q),
                                       ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_attn_decode_step")
    return out, lse


def path_attn_chunk_size(d: int, dtype_code: int) -> int:
    c = load_library().path_attn_chunk_size(d, dtype_code)
    if c < 0:
        raise PathAttnError(c, "path_attn_chunk_size")
    return c


def path_attn_debug_factors(q, k, w, beta, logf=None, scale=None, stream=None):
    """Chunk factors of the preparation step (diagnostics; see the header)."""
    import torch
    lib = load_library()
    _check_inputs(q, k, q, w, beta, logf, True)
    B, H, T, d = q.shape
    if scale is None:
        scale = d ** -0.5
    code = _dtype_code(q)
    C = path_attn_chunk_size(d, code)
    Np = -(-T // C)
    BH, Tp = B * H, Np * C
    dev = q.device
    kr = torch.empty((BH, Tp, d), device=dev, dtype=q.dtype)
    ql = torch.empty((BH, Tp, d), device=dev, dtype=torch.float32)
    ngt = torch.empty((BH, Np, d, d), device=dev, dtype=q.dtype)
    sdt = torch.empty((BH, Np, C, C), device=dev, dtype=torch.float32)
    lam2 = torch.empty((BH, Tp), device=dev, dtype=torch.float32) if logf is not None else None
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.path_attn_debug_factors(_ptr(q), _ptr(k), _ptr(w), _ptr(beta), _ptr(logf),
                                         float(scale), B, H, T, d, code, _ptr(kr), _ptr(ql),
                                         _ptr(ngt), _ptr(sdt), _ptr(lam2),
                                         ctypes.c_void_p(st.cuda_stream))
    _check(rc, "path_attn_debug_factors")
    return dict(C=C, kr=kr, ql=ql, ngt=ngt, sdt=sdt, lam2=lam2)


def path_attn_debug_wait_timeout(limit_ns: int, stream=None):
    """Launch the diagnostics kernel whose bounded wait expires after
    ``limit_ns``; the device status word then reads PATH_ERR_TIMEOUT."""
    import torch
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(load_library().path_attn_debug_wait_timeout(int(limit_ns), ctypes.c_void_p(st.cuda_stream)),
           "path_attn_debug_wait_timeout")


def path_attn_device_status(device: int = 0, clear: bool = True) -> int:
    """0 if no kernel reported an error on ``device`` since the last clear,
    else a negative status: PATH_ERR_TIMEOUT (a bounded wait expired) or
    PATH_ERR_INVALID_ARG (a decoding position out of bounds).  Synchronises
    the device."""
    return load_library().path_attn_device_status(device, 1 if clear else 0)


def path_attn_workspace_bytes(B, H, T, d, dtype_code, with_gate=False) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().path_attn_workspace_bytes(B, H, T, d, dtype_code, int(with_gate),
                                                    ctypes.byref(n)),
           "path_attn_workspace_bytes")
    return n.value


def path_attn_launches_per_call(d, dtype_code, with_gate=False) -> int:
    n = load_library().path_attn_launches_per_call(d, dtype_code, int(with_gate))
    if n < 0:
        raise PathAttnError(n, "path_attn_launches_per_call")
    return n


def path_attn_set_transition_form(form: int = 0):
    """0: dense transitions (default); 1: the low-rank form q <- q - (q W^T)(U W)
    for bf16 problems at d = 64 (others keep the dense form)."""
    _check(load_library().path_attn_set_transition_form(int(form)),
           "path_attn_set_transition_form")


def path_attn_timing_enable(enable: bool = True):
    _check(load_library().path_attn_timing_enable(1 if enable else 0), "path_attn_timing_enable")


def path_attn_timing_read():
    """(prep_ms_total, attn_ms_total, calls) since timing was enabled."""
    p, a, c = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_long(0)
    _check(load_library().path_attn_timing_read(ctypes.byref(p), ctypes.byref(a), ctypes.byref(c)),
           "path_attn_timing_read")
    return p.value, a.value, c.value


BWD_PHASES = ("prep", "rowdot", "xwalk", "key", "gwalk", "dF", "chunk")


def path_attn_bwd_timing_read():
    """({phase: ms_total}, calls) of path_attn_bwd since timing was enabled;
    phases in launch order (``BWD_PHASES``)."""
    ms = (ctypes.c_double * len(BWD_PHASES))()
    c = ctypes.c_long(0)
    _check(load_library().path_attn_bwd_timing_read(ms, ctypes.byref(c)),
           "path_attn_bwd_timing_read")
    return dict(zip(BWD_PHASES, list(ms))), c.value


def path_attn_version() -> int:
    return load_library().path_attn_version()


def path_attn_status_string(status: int) -> str:
    return load_library().path_attn_status_string(status).decode()
