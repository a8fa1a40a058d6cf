"""The allocation-free entry point, path_attn_fwd_noalloc.

It serves callers that may not allocate device memory (a host framework that
has reserved the device's memory for its own allocator, or a serving loop with
a fixed memory budget): its workspace is a static device array inside the
library.  These tests call it through the C ABI and compare it with
path_attn_fwd on the same inputs, two calls in a row, with the tolerances of
the other GPU tests.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import householder_softmax_attention_gb300 as pa
from seeded_inputs import Workload, make_inputs

TOL_F32 = 1e-4
TOL_BF16_ABS = 2e-2
TOL_BF16_REL = 5e-3
UNSUPPORTED = -2


@pytest.fixture(scope="module")
def lib():
    from householder_softmax_attention_gb300 import build
    build.build()
    return pa.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, x, status):
    q, k, v, w, beta, logf = (x[n] for n in ("q", "k", "v", "w", "beta", "logf"))
    B, H, T, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    code = pa.PATH_DTYPE_BF16 if q.dtype == torch.bfloat16 else pa.PATH_DTYPE_F32
    rc = lib.path_attn_fwd_noalloc(_p(q), _p(k), _p(v), _p(w), _p(beta), _p(logf),
                                   float(x["scale"]), _p(out), _p(lse), _p(status),
                                   B, H, T, d, code,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, pa.path_attn_status_string(rc)
    return out, lse


def _close(a, b, bf16):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    err = np.abs(a - b)
    if bf16:
        assert err.max() <= TOL_BF16_ABS
        assert err.sum() <= TOL_BF16_REL * np.abs(b).sum()
    else:
        assert err.max() <= TOL_F32


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_two_calls_in_a_row(lib):
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    cases = [Workload("noalloc_a", 1, 2, 1000, 128, "bf16", fox=True, seed=31),
             Workload("noalloc_b", 2, 1, 333, 64, "bf16", seed=32),
             Workload("noalloc_c", 1, 2, 200, 64, "f32", seed=33)]
    for wl in cases:
        x = {n: (t.cuda() if torch.is_tensor(t) else t) for n, t in make_inputs(wl).items()}
        ref_out, ref_lse = pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"],
                                            x["logf"], x["scale"])
        for _ in range(2):  # the shared scratch keeps the previous call's contents
            out, lse = _noalloc(lib, x, status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            bf = wl.dtype == "bf16"
            _close(out, ref_out, bf)
            _close(lse, ref_lse, bf)


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_the_static_scratch(lib):
    wl = Workload("noalloc_big", 2, 16, 4096, 128, "bf16", seed=34)
    need = pa.path_attn_workspace_bytes(wl.B, wl.H, wl.T, wl.d, pa.PATH_DTYPE_BF16)
    assert need > 64 << 20
    x = {n: (t.cuda() if torch.is_tensor(t) else t) for n, t in make_inputs(wl).items()}
    q = x["q"]
    out = torch.empty_like(q)
    rc = lib.path_attn_fwd_noalloc(_p(q), _p(x["k"]), _p(x["v"]), _p(x["w"]), _p(x["beta"]),
                                   None, float(x["scale"]), _p(out), None, None,
                                   wl.B, wl.H, wl.T, wl.d, pa.PATH_DTYPE_BF16, None)
    assert rc == UNSUPPORTED
    assert b"workspace" in lib.path_attn_last_error()


@pytest.mark.gpu
def test_noalloc_null_status_is_readable(lib):
    """With status NULL the kernels report into the library's static word;
    path_attn_noalloc_status reads it (0 after a call whose waits all ended)
    and clears it, allocating nothing."""
    wl = Workload("noalloc_null", 1, 2, 300, 128, "bf16", seed=35)
    x = {n: (t.cuda() if torch.is_tensor(t) else t) for n, t in make_inputs(wl).items()}
    ref_out, _ = pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, x["scale"])
    for _ in range(2):
        out, _ = _noalloc(lib, x, None)
        assert lib.path_attn_noalloc_status(0, 1) == 0
        _close(out, ref_out, True)
    assert pa.path_attn_noalloc_status(0, False) == 0
