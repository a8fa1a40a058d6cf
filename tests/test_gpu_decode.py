"""GPU parity of decoding with keys rewritten in place (slides' frame
"Decoding updates historical keys in place"): the prefill cache, token-by-token
decoding after a prefill, ragged batch positions, the empty-cache start, the
device-side position check, and one full-size step on a 16K cache.

Expected values come only from the fp64 oracle (``path_oracle_fwd``,
``path_oracle_decoded_keys``, ``path_oracle_decode_step``).
Tolerances: fp32 inputs 1e-4 max-abs on out and lse; bf16 inputs 2e-2 max-abs
and 5e-3 mean-relative on out, 2e-2 max-abs on lse (as for the forward).
"""
import numpy as np
import pytest
import torch

import householder_softmax_attention_gb300 as pa
from oracle import path_oracle_decode_step, path_oracle_decoded_keys, path_oracle_fwd
from seeded_inputs import DECODE_WORKLOADS, Workload, make_decode_inputs, make_inputs

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _check_out(out, ref, lse, ref_lse, bf16, what):
    err = np.abs(out - ref)
    if bf16:
        assert err.max() <= 2e-2, f"{what}: out max-abs {err.max():.3e}"
        mrel = err.sum() / np.abs(ref).sum()
        assert mrel <= 5e-3, f"{what}: out mean-rel {mrel:.3e}"
        assert np.abs(lse - ref_lse).max() <= 2e-2, f"{what}: lse"
    else:
        assert err.max() <= 1e-4, f"{what}: out max-abs {err.max():.3e}"
        assert np.abs(lse - ref_lse).max() <= 1e-4, f"{what}: lse"


def _key_tol(ref, bf16):
    # bf16 prefill builds the cache from bf16-rounded chunk factors (2^-9
    # relative each, a few transitions deep); fp32 from fp32 factors
    return (2e-4 + 2 ** -7 * np.abs(ref).max()) if bf16 else 2e-4


CASES = [("f32", 64, False), ("f32", 128, True), ("bf16", 128, False), ("bf16", 128, True),
         ("bf16", 64, True)]


@pytest.mark.parametrize("dtype,d,fox", CASES)
def test_prefill_fills_cache_with_keys_carried_to_the_prompt_end(dtype, d, fox):
    wl = Workload("prefill", 1, 2, 300, d, dtype, fox=fox, seed=31)
    x = make_inputs(wl)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    Tmax = 333
    cache = pa.DecodeCache(1, 2, Tmax, d, wl.torch_dtype, "cuda", gated=fox)
    cache.kcache.fill_(7.0)
    cache.vcache.fill_(7.0)
    out, lse = pa.path_attn_prefill(dev["q"], dev["k"], dev["v"], dev["w"], dev["beta"],
                                    dev["logf"], cache, scale=x["scale"])
    ref_out, ref_lse = pa.path_attn_fwd(dev["q"], dev["k"], dev["v"], dev["w"], dev["beta"],
                                        dev["logf"], scale=x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    bf = dtype == "bf16"
    for h in range(2):
        k, w = _np(x["k"])[0, h], _np(x["w"])[0, h]
        beta = _np(x["beta"])[0, h]
        ref = path_oracle_decoded_keys(k, w, beta, wl.T - 1)
        got = _np(cache.kcache)[0, h, : wl.T]
        np.testing.assert_allclose(got, ref, atol=_key_tol(ref, bf), rtol=0)
    assert torch.equal(cache.vcache[:, :, : wl.T], dev["v"])
    assert torch.all(cache.kcache[:, :, wl.T:] == 7.0) and torch.all(cache.vcache[:, :, wl.T:] == 7.0)
    if fox:
        lam = np.cumsum(_np(x["logf"]), axis=-1)
        np.testing.assert_allclose(_np(cache.lamcache)[:, :, : wl.T], lam, atol=2e-5, rtol=1e-6)


def _step_inputs(x, t):
    sl = lambda n: x[n][:, :, t].contiguous().cuda()
    return (sl("q"), sl("k"), sl("v"), sl("w"), sl("beta"),
            None if x["logf"] is None else sl("logf"))


@pytest.mark.parametrize("dtype,d,fox", CASES)
def test_decoding_after_prefill_matches_the_forward_rows(dtype, d, fox):
    """Prefill P tokens, decode the rest one at a time: every decoded row is
    row t of the oracle forward over the whole sequence."""
    P, T = 200, 264
    wl = Workload("decode", 1, 2, T, d, dtype, fox=fox, seed=32)
    x = make_inputs(wl)
    pref = {n: (x[n][:, :, :P].contiguous().cuda() if x[n] is not None else None)
            for n in ("q", "k", "v", "w", "beta", "logf")}
    cache = pa.DecodeCache(1, 2, T, d, wl.torch_dtype, "cuda", gated=fox)
    pa.path_attn_prefill(pref["q"], pref["k"], pref["v"], pref["w"], pref["beta"],
                         pref["logf"], cache, scale=x["scale"])
    outs, lses = [], []
    for t in range(P, T):
        pos = torch.full((1,), t, dtype=torch.int32, device="cuda")
        q, k, v, w, b, lf = _step_inputs(x, t)
        o, l = pa.path_attn_decode_step(q, k, v, w, b, lf, cache, pos, T, scale=x["scale"])
        outs.append(o.clone())
        lses.append(l.clone())
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, clear=True) == 0
    got = np.stack([_np(o) for o in outs], axis=2)      # [1, 2, T-P, d]
    got_lse = np.stack([_np(l) for l in lses], axis=2)  # [1, 2, T-P]
    bf = dtype == "bf16"
    for h in range(2):
        arr = {n: _np(x[n])[0, h] for n in ("q", "k", "v", "w", "beta")}
        lf = None if x["logf"] is None else _np(x["logf"])[0, h]
        rows = np.arange(P, T)
        ref, ref_lse = path_oracle_fwd(arr["q"], arr["k"], arr["v"], arr["w"], arr["beta"],
                                       logf=lf, scale=x["scale"], rows=rows)
        _check_out(got[0, h], ref, got_lse[0, h], ref_lse, bf, f"head {h}")
        keys = path_oracle_decoded_keys(arr["k"], arr["w"], arr["beta"], T - 1)
        np.testing.assert_allclose(_np(cache.kcache)[0, h], keys, atol=_key_tol(keys, bf), rtol=0)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_decoding_from_an_empty_cache(dtype, d):
    T = 70
    wl = Workload("decode0", 1, 1, T, d, dtype, seed=33)
    x = make_inputs(wl)
    cache = pa.DecodeCache(1, 1, T, d, wl.torch_dtype, "cuda")
    outs = []
    for t in range(T):
        pos = torch.full((1,), t, dtype=torch.int32, device="cuda")
        q, k, v, w, b, _ = _step_inputs(x, t)
        o, l = pa.path_attn_decode_step(q, k, v, w, b, None, cache, pos, max_len=t + 1,
                                        scale=x["scale"])
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    got = np.stack([_np(o)[0, 0] for o, _ in outs])
    got_lse = np.array([_np(l)[0, 0] for _, l in outs])
    arr = {n: _np(x[n])[0, 0] for n in ("q", "k", "v", "w", "beta")}
    ref, ref_lse = path_oracle_fwd(arr["q"], arr["k"], arr["v"], arr["w"], arr["beta"],
                                   scale=x["scale"])
    _check_out(got, ref, got_lse, ref_lse, dtype == "bf16", "empty-cache decode")
    # token 0 attends to itself only
    np.testing.assert_allclose(got[0], arr["v"][0], atol=1e-6 if dtype == "f32" else 1e-2)


def _oracle_step(x, b, h, t, dtype):
    """The oracle's decoding step of (b, h) at position t over the drawn cache."""
    kc = np.ascontiguousarray(_np(x["kcache"][b, h, : t + 1]))
    vc = np.ascontiguousarray(_np(x["vcache"][b, h, : t + 1]))
    lam = None if x["lamcache"] is None else np.ascontiguousarray(_np(x["lamcache"][b, h, : t + 1]))
    g = lambda n: _np(x[n])[b, h]
    lf = None if x["logf"] is None else float(_np(x["logf"])[b, h])
    o, l = path_oracle_decode_step(kc, vc, lam, g("q"), g("k"), g("v"), g("w"),
                                   float(_np(x["beta"])[b, h]), lf, t, scale=x["scale"])
    return o, l, kc, lam


@pytest.mark.parametrize("fox", [False, True])
def test_ragged_positions_and_position_check(fox):
    """Batch rows at different positions; then a position outside its bound
    is refused on the device without touching that row's cache."""
    wl = Workload("ragged", 3, 2, 700, 128, "bf16", fox=fox, seed=34)
    x = make_decode_inputs(wl)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    cache = pa.DecodeCache.wrap(dev["kcache"].clone(), dev["vcache"].clone(),
                                None if dev["lamcache"] is None else dev["lamcache"].clone())
    pos_h = [699, 0, 313]
    pos = torch.tensor(pos_h, dtype=torch.int32, device="cuda")
    out, lse = pa.path_attn_decode_step(dev["q"], dev["k"], dev["v"], dev["w"], dev["beta"],
                                        dev["logf"], cache, pos, max_len=700, scale=x["scale"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, clear=True) == 0
    for b in range(3):
        t = pos_h[b]
        for h in range(2):
            o, l, kc, lam = _oracle_step(x, b, h, t, "bf16")
            _check_out(_np(out)[b, h][None], o[None], _np(lse)[b, h][None], np.array([l]),
                       True, f"b{b} h{h}")
            np.testing.assert_allclose(_np(cache.kcache)[b, h, : t + 1], kc, atol=1e-5, rtol=1e-5)
            if lam is not None:
                np.testing.assert_allclose(_np(cache.lamcache)[b, h, : t + 1], lam, atol=1e-5)
            # rows past the new token are untouched
            assert torch.equal(cache.kcache[b, h, t + 1:], dev["kcache"][b, h, t + 1:])
    # an out-of-range position: NaN for that row, status INVALID_ARG, cache kept
    before = cache.kcache.clone()
    bad = torch.tensor([5, 700, 6], dtype=torch.int32, device="cuda")
    out, lse = pa.path_attn_decode_step(dev["q"], dev["k"], dev["v"], dev["w"], dev["beta"],
                                        dev["logf"], cache, bad, max_len=700, scale=x["scale"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, clear=True) == -1  # PATH_ERR_INVALID_ARG
    assert torch.isnan(out[1]).all() and torch.isnan(lse[1]).all()
    assert torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all()
    assert torch.equal(cache.kcache[1], before[1])
    assert pa.path_attn_device_status(0, clear=True) == 0


@pytest.mark.parametrize("name", sorted(DECODE_WORKLOADS))
def test_full_size_decode_step_sampled(name):
    """One step at position T - 1 of a full 16K cache (the benchmarked launch
    configuration), checked on sampled heads against the oracle's step."""
    wl = DECODE_WORKLOADS[name]
    x = make_decode_inputs(wl, device="cuda")
    x_cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in x.items()}
    cache = pa.DecodeCache.wrap(x["kcache"].clone(), x["vcache"].clone())
    T = wl.T
    pos = torch.full((wl.B,), T - 1, dtype=torch.int32, device="cuda")
    out, lse = pa.path_attn_decode_step(x["q"], x["k"], x["v"], x["w"], x["beta"], None, cache,
                                        pos, max_len=T, scale=x["scale"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, clear=True) == 0
    for b, h in ((0, 0), (wl.B - 1, wl.H - 1), (wl.B - 1, 3)):
        o, l, kc, _ = _oracle_step(x_cpu, b, h, T - 1, "bf16")
        _check_out(_np(out)[b, h][None], o[None], _np(lse)[b, h][None], np.array([l]), True,
                   f"{name} b{b} h{h}")
        got = _np(cache.kcache[b, h])
        np.testing.assert_allclose(got, kc, atol=2e-5, rtol=1e-5)
