"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and its host-side logic (sizes, validation, status strings)
behaves as documented.  No call here reaches a CUDA kernel."""
import ctypes
import re

import pytest

import householder_softmax_attention_gb300 as pa
from householder_softmax_attention_gb300 import build as pa_build

PATH_OK, INVALID, UNSUPPORTED = 0, -1, -2


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pa.load_library()


def _declared_symbols():
    text = open(pa.HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(path_attn_\w+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = _declared_symbols()
    assert "path_attn_fwd" in names and "path_attn_fwd_host" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pathattn.h but not exported"


def test_status_strings_and_version(lib):
    assert pa.path_attn_status_string(0) == "PATH_OK"
    assert pa.path_attn_status_string(-4) == "PATH_ERR_TIMEOUT"
    assert pa.path_attn_status_string(-99) == "PATH_ERR_UNKNOWN"
    assert pa.path_attn_version() >= 100


def test_chunk_size_and_launch_count(lib):
    assert pa.path_attn_chunk_size(128, pa.PATH_DTYPE_BF16) == 128
    assert pa.path_attn_chunk_size(64, pa.PATH_DTYPE_F32) == 64
    assert lib.path_attn_chunk_size(96, pa.PATH_DTYPE_BF16) == UNSUPPORTED
    assert lib.path_attn_chunk_size(64, 7) == INVALID
    n0 = pa.path_attn_launches_per_call(128, pa.PATH_DTYPE_BF16, False)
    n1 = pa.path_attn_launches_per_call(128, pa.PATH_DTYPE_BF16, True)
    assert n1 == n0 + 1 and n0 >= 2


def test_workspace_bytes_grow_with_problem(lib):
    a = pa.path_attn_workspace_bytes(1, 2, 256, 64, pa.PATH_DTYPE_F32)
    b = pa.path_attn_workspace_bytes(1, 2, 512, 64, pa.PATH_DTYPE_F32)
    c = pa.path_attn_workspace_bytes(1, 2, 512, 64, pa.PATH_DTYPE_F32, with_gate=True)
    assert 0 < a < b < c
    # a ragged length takes the same chunks as the next multiple of the chunk
    assert pa.path_attn_workspace_bytes(2, 16, 1000, 128, pa.PATH_DTYPE_BF16) == \
        pa.path_attn_workspace_bytes(2, 16, 1024, 128, pa.PATH_DTYPE_BF16)
    n = ctypes.c_size_t(0)
    assert lib.path_attn_workspace_bytes(0, 1, 1, 64, 1, 0, ctypes.byref(n)) == INVALID
    assert lib.path_attn_workspace_bytes(1, 1, 1, 80, 1, 0, ctypes.byref(n)) == UNSUPPORTED
    assert lib.path_attn_workspace_bytes(1, 1, 1, 64, 1, 0, None) == INVALID
    # index space overflow is refused, not wrapped
    assert lib.path_attn_workspace_bytes(4096, 4096, 65536, 128, 1, 0, ctypes.byref(n)) == UNSUPPORTED


def _fwd(lib, ptrs, B=1, H=1, T=8, d=64, dtype=1, logf=None, lse=None, scale=0.125):
    q, k, v, w, beta, out = ptrs
    return lib.path_attn_fwd(q, k, v, w, beta, logf, scale, out, lse, B, H, T, d, dtype, None)


def test_validation_happens_before_any_cuda_call(lib):
    good = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(6)]
    # NULL required pointers
    for i in range(6):
        ptrs = list(good)
        ptrs[i] = None
        assert _fwd(lib, ptrs) == INVALID
    # misaligned pointers
    for i in range(6):
        ptrs = list(good)
        ptrs[i] = ctypes.c_void_p(0x10008 + 0x10000 * i)
        assert _fwd(lib, ptrs) == INVALID
    assert _fwd(lib, good, logf=ctypes.c_void_p(0x70004)) == INVALID
    # sizes and dtype
    assert _fwd(lib, good, T=0) == INVALID
    assert _fwd(lib, good, B=-1) == INVALID
    assert _fwd(lib, good, d=32) == UNSUPPORTED
    assert _fwd(lib, good, dtype=5) == INVALID
    assert _fwd(lib, good, scale=float("nan")) == INVALID
    # the host-buffer entry checks the same sizes first
    q, k, v, w, beta, out = good
    assert lib.path_attn_fwd_host(q, k, v, w, beta, None, 0.1, out, None, 1, 1, 0, 64, 1,
                                  None) == INVALID
    assert lib.path_attn_debug_factors(q, k, w, beta, None, 0.1, 1, 1, 8, 64, 1, None, None,
                                       None, None, None, None) == INVALID


def test_decode_and_prefill_validate_before_any_cuda_call(lib):
    g = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(12)]
    q, k, v, w, beta, out, kc, vc, pos = g[:9]
    lam, logf = g[9], g[10]
    dec = lambda **kw: lib.path_attn_decode_step(
        kw.get("q", q), k, v, w, beta, kw.get("logf"), kw.get("scale", 0.1), kw.get("kc", kc), vc,
        kw.get("lam"), kw.get("pos", pos), kw.get("max_len", 8), out, None, 1, 1,
        kw.get("Tmax", 8), kw.get("d", 64), 1, None)
    assert dec(q=None) == INVALID
    assert dec(pos=None) == INVALID
    assert dec(kc=ctypes.c_void_p(0x70008)) == INVALID      # misaligned cache
    assert dec(logf=logf) == INVALID                        # gate without its prefix cache
    assert dec(lam=lam) == INVALID                          # prefix cache without a gate
    assert dec(max_len=9) == INVALID                        # above Tmax
    assert dec(max_len=0) == INVALID
    assert dec(d=96) == UNSUPPORTED
    assert dec(scale=float("nan")) == INVALID
    pre = lambda **kw: lib.path_attn_prefill(
        q, k, v, w, beta, kw.get("logf"), 0.1, out, None, kw.get("kc", kc), vc, kw.get("lam"),
        kw.get("Tmax", 16), 1, 1, kw.get("T", 16), 64, 1, None)
    assert pre(kc=None) == INVALID
    assert pre(Tmax=15) == INVALID                          # cache shorter than the prompt
    assert pre(logf=logf) == INVALID
    assert pre(T=0) == INVALID


def test_partial_validates_before_any_cuda_call(lib):
    q, k, v, w, beta, out = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(6)]
    part = lambda r, w=w, d=64: lib.path_attn_fwd_partial(q, k, v, w, beta, None, 0.1, out, None,
                                                         1, 1, 8, d, r, 1, None)
    assert part(65) == INVALID          # r above d
    assert part(-1) == INVALID
    assert part(8, w=None) == INVALID   # u needed when r > 0
    assert part(0, d=96) == UNSUPPORTED


def test_producer_validates_before_any_cuda_call(lib):
    p = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    prod = lambda B=1, T=8, Dm=128, H=2, d=64, R=16, dt=1, ptrs=p: lib.path_producer_fwd(
        *ptrs, B, T, Dm, H, d, R, dt, None)
    assert prod(Dm=100) == UNSUPPORTED       # Dm not a multiple of 64
    assert prod(R=24) == UNSUPPORTED         # R not a multiple of 16
    assert prod(R=128, H=8) == UNSUPPORTED   # R + H above 128
    assert prod(d=96) == UNSUPPORTED
    assert prod(T=0) == INVALID
    assert prod(dt=4) == INVALID
    bad = list(p)
    bad[0] = None
    assert prod(ptrs=bad) == INVALID
    bad = list(p)
    bad[6] = ctypes.c_void_p(0x70008)        # misaligned w
    assert prod(ptrs=bad) == INVALID


def test_backward_launch_count(lib):
    bf, f32 = pa.PATH_DTYPE_BF16, pa.PATH_DTYPE_F32
    one = pa.path_attn_bwd_launches_per_call(128, 128, bf)     # one chunk: no X walk
    many = pa.path_attn_bwd_launches_per_call(4096, 128, bf)
    assert many == one + 1
    # the gate adds its prefix sum and its suffix scan
    assert pa.path_attn_bwd_launches_per_call(4096, 128, bf, True) == many + 2
    assert pa.path_attn_bwd_launches_per_call(300, 64, f32) > many
    assert lib.path_attn_bwd_launches_per_call(0, 128, bf, 0) == INVALID
    assert lib.path_attn_bwd_launches_per_call(64, 96, bf, 0) == UNSUPPORTED


def test_backward_timing_read_without_calls(lib):
    pa.path_attn_timing_enable(True)
    phases, calls = pa.path_attn_bwd_timing_read()
    pa.path_attn_timing_enable(False)
    assert calls == 0 and set(phases) == set(pa.BWD_PHASES)
    assert all(v == 0.0 for v in phases.values())
