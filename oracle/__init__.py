"""CPU oracle for the PaTH attention forward pass -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never does, and this package never imports the product.

Two independent formulations live here, both in fp64:

* ``path_oracle_fwd`` / ``path_oracle_logits`` -- the literal definition in C
  (``path_oracle.c``): for each query, propagate ``z = q_i`` backward through
  ``H_i, H_{i-1}, ...`` and emit every logit, then an exact causal softmax.
  Source: "PaTH Attention: Position Encoding via Accumulating Householder
  Transformations" (slides), frames "PaTH inserts a learned transformation
  along every path" and "FoX adds a separate mechanism for forgetting".
* ``path_oracle_decoded_keys`` / ``path_oracle_decode_step`` -- decoding with
  keys rewritten in place (frame "Decoding updates historical keys in place"),
  also in C.
* ``path_oracle_partial_fwd`` -- partial PaTH (PaTH on the first r head
  dimensions, no position encoding on the rest), in C.
* ``chunked`` -- the blockwise UT-transform algebra in numpy (frames "A
  triangular representation makes paths computable", "A right-to-left scan
  accumulates cross-block paths" and "Backup: fix orientation before
  implementing UT products").  It is pinned against the literal definition and
  supplies the expected chunk factors for the GPU factor tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "path_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libpath_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into ``oracle/_build``; return the path."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            lib.path_oracle_fwd.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, dp,
                ctypes.c_double, ctypes.c_long, lp, dp, dp, ctypes.c_int]
            lib.path_oracle_fwd.restype = ctypes.c_int
            lib.path_oracle_logits.argtypes = [
                ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, ctypes.c_double,
                ctypes.c_int, dp]
            lib.path_oracle_logits.restype = ctypes.c_int
            lib.path_oracle_decoded_keys.argtypes = [
                ctypes.c_int, ctypes.c_int, dp, dp, dp, ctypes.c_int, dp]
            lib.path_oracle_decoded_keys.restype = ctypes.c_int
            lib.path_oracle_decode_step.argtypes = [
                ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, dp, dp, ctypes.c_double,
                dp, ctypes.c_double, dp, dp]
            lib.path_oracle_decode_step.restype = ctypes.c_int
            lib.path_oracle_partial_fwd.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, dp,
                ctypes.c_double, dp, dp]
            lib.path_oracle_partial_fwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def path_oracle_fwd(q, k, v, w, beta, logf=None, scale=None, rows=None,
                    threads=None):
    """Literal PaTH(-FoX) forward in fp64.

    q, k, v, w: ``[..., T, d]`` (any leading batch/head dims, flattened to BH);
    beta, logf: ``[..., T]``.  ``scale`` defaults to ``1/sqrt(d)``.
    ``rows``: optional flat row ids ``bh*T + i``; then ``out`` is
    ``[len(rows), d]`` and ``lse`` ``[len(rows)]``.  Otherwise ``out`` has the
    shape of ``q`` and ``lse`` the shape of ``beta``.
    Inputs are converted to fp64 exactly as stored (a bf16 tensor is widened,
    not re-rounded).
    """
    q, k, v, w, beta = (_f64(x) for x in (q, k, v, w, beta))
    lf = None if logf is None else _f64(logf)
    *lead, T, d = q.shape
    BH = int(np.prod(lead)) if lead else 1
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    for x in (k, v, w):
        assert x.shape == q.shape, "q, k, v, w must share one shape"
    assert beta.shape == q.shape[:-1]
    if lf is not None:
        assert lf.shape == beta.shape
    if rows is None:
        n = BH * T
        rp = None
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = int(rows.size)
        rp = rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().path_oracle_fwd(BH, T, d, _ptr(q), _ptr(k), _ptr(v), _ptr(w),
                                 _ptr(beta), _ptr(lf), float(scale), n, rp,
                                 _ptr(out), _ptr(lse),
                                 int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"path_oracle_fwd failed with status {rc}")
    if rows is None:
        return out.reshape(q.shape), lse.reshape(beta.shape)
    return out, lse


def path_oracle_logits(q, k, w, beta, i, logf=None, scale=None):
    """Log-weights ``scale * k_j^T H_{j+1}..H_i q_i + gate_ij`` for j = 0..i of
    one head (q, k, w: ``[T, d]``; beta, logf: ``[T]``)."""
    q, k, w, beta = (_f64(x) for x in (q, k, w, beta))
    lf = None if logf is None else _f64(logf)
    T, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    s = np.zeros((i + 1,), dtype=np.float64)
    rc = _load().path_oracle_logits(T, d, _ptr(q), _ptr(k), _ptr(w), _ptr(beta),
                                    _ptr(lf), float(scale), int(i), _ptr(s))
    if rc != 0:
        raise RuntimeError(f"path_oracle_logits failed with status {rc}")
    return s


def path_oracle_decoded_keys(k, w, beta, t):
    """Keys of one head (``k, w: [T, d]``, ``beta: [T]``) as a decoder holds
    them after token ``t``: ``k_j^(t) = H_t ... H_{j+1} k_j`` for j < t and
    ``k_t``; returns ``[t + 1, d]``."""
    k, w, beta = (_f64(x) for x in (k, w, beta))
    T, d = k.shape
    out = np.zeros((t + 1, d), dtype=np.float64)
    rc = _load().path_oracle_decoded_keys(T, d, _ptr(k), _ptr(w), _ptr(beta), int(t), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"path_oracle_decoded_keys failed with status {rc}")
    return out


def path_oracle_decode_step(kc, vc, lam, q, k, v, w, beta, logf, t, scale=None):
    """One decoding step of one head at position ``t``.

    ``kc, vc``: ``[>= t + 1, d]`` fp64 arrays, rows ``< t`` hold the cache and
    are rewritten in place, row ``t`` receives ``k`` / ``v``; ``lam``:
    ``[>= t + 1]`` gate prefixes (natural log) or None with ``logf`` None.
    Returns ``(out [d], lse)``.
    """
    for a in (kc, vc) + (() if lam is None else (lam,)):
        assert a.dtype == np.float64 and a.flags.c_contiguous
    q, k, v, w = (_f64(x) for x in (q, k, v, w))
    d = q.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    lf = None if logf is None else np.array([float(logf)], dtype=np.float64)
    out = np.zeros(d)
    lse = np.zeros(1)
    rc = _load().path_oracle_decode_step(int(t), d, _ptr(kc), _ptr(vc), _ptr(lam), _ptr(q),
                                         _ptr(k), _ptr(v), _ptr(w), float(beta), _ptr(lf),
                                         float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"path_oracle_decode_step failed with status {rc}")
    return out, float(lse[0])


def path_oracle_partial_fwd(q, k, v, u, beta, logf=None, scale=None):
    """Partial PaTH forward in fp64: PaTH with ``u [..., T, r]`` on the first
    ``r`` head dimensions, plain dot products on the other ``d - r``.  Shapes
    as ``path_oracle_fwd`` (``u`` has its own last dimension r, 0 <= r <= d).
    Returns ``(out, lse)``."""
    q, k, v, beta = (_f64(x) for x in (q, k, v, beta))
    u = _f64(u)
    lf = None if logf is None else _f64(logf)
    *lead, T, d = q.shape
    r = u.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((BH * T, d))
    lse = np.zeros(BH * T)
    rc = _load().path_oracle_partial_fwd(BH, T, d, r, _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(u) if r > 0 else None, _ptr(beta), _ptr(lf),
                                         float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"path_oracle_partial_fwd failed with status {rc}")
    return out.reshape(q.shape), lse.reshape(beta.shape)
