"""Pins for the fp64 CPU oracle: checks against what the PaTH pages and plain
mathematics fix, so that a dropped term, a wrong sign or index, or a reversed
product order in the oracle fails at least one test.

Sources ("PaTH Attention: Position Encoding via Accumulating Householder
Transformations", discussion slides):
  * frame "PaTH inserts a learned transformation along every path" (definition)
  * frame "One direction can shrink, disappear, or change sign" (eigen-action)
  * frame "PaTH keeps a recurrent path and a softmax readout" (linear RNN view)
  * frame "A reflection can implement a symbolic swap"
  * frame "FoX adds a separate mechanism for forgetting"
  * frame "Backup: two heads distinguish the identity permutation"
"""
import math
import os
import re

import numpy as np
import pytest
import torch

from oracle import (path_oracle_decode_step, path_oracle_decoded_keys, path_oracle_fwd,
                    path_oracle_logits, path_oracle_partial_fwd)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, T, d, beta="sig", unit=True):
    q = rng.standard_normal((T, d))
    k = rng.standard_normal((T, d))
    v = rng.standard_normal((T, d))
    w = rng.standard_normal((T, d))
    if unit:
        w /= np.linalg.norm(w, axis=1, keepdims=True)
    if beta == "sig":
        b = 2.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    else:
        b = np.full(T, float(beta))
    return q, k, v, w, b


def _causal_softmax_attention(q, k, v, scale):
    """Plain causal softmax attention, written out independently."""
    T = q.shape[0]
    out = np.zeros_like(v)
    lse = np.zeros(T)
    for i in range(T):
        s = scale * (k[: i + 1] @ q[i])
        m = s.max()
        p = np.exp(s - m)
        out[i] = p @ v[: i + 1] / p.sum()
        lse[i] = m + math.log(p.sum())
    return out, lse


# ---------------------------------------------------------------- I1: beta = 0
@pytest.mark.parametrize("zero", ["beta", "w"])
def test_beta_or_w_zero_is_causal_softmax_attention(zero):
    rng = np.random.default_rng(1)
    T, d = 40, 16
    q, k, v, w, b = _rand_inputs(rng, T, d)
    if zero == "beta":
        b[:] = 0.0
    else:
        w[:] = 0.0
    scale = 0.37
    out, lse = path_oracle_fwd(q, k, v, w, b, scale=scale)
    ref_out, ref_lse = _causal_softmax_attention(q, k, v, scale)
    np.testing.assert_allclose(out, ref_out, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-13, rtol=0)
    # and against the library routine, in fp64 on the CPU
    t = lambda x: torch.from_numpy(x)[None, None]
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), is_causal=True, scale=scale)[0, 0].numpy()
    np.testing.assert_allclose(out, sdpa, atol=1e-12, rtol=0)


# ---------------------------------------------------- eigen-action (golden)
def _read_eigen():
    rows = []
    with open(os.path.join(GOLDEN, "eigen_action.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                b, along, orth, _ = line.split()
                rows.append((float(b), float(along), float(orth)))
    return rows


@pytest.mark.parametrize("beta,along,orth", _read_eigen())
def test_eigen_action_of_one_transition(beta, along, orth):
    # Two tokens; the logit of query 1 against key 0 is k_0^T H_1 q_1.
    rng = np.random.default_rng(2)
    d = 6
    w1 = rng.standard_normal(d)
    w1 /= np.linalg.norm(w1)
    perp = rng.standard_normal(d)
    perp -= (perp @ w1) * w1
    alpha = 0.8
    q1 = perp + alpha * w1
    q = np.stack([np.zeros(d), q1])
    w = np.stack([np.zeros(d), w1])
    b = np.array([0.0, beta])
    # key along w reads the w-component, key along perp the orthogonal part
    for key, expect in ((w1, along * alpha),
                        (perp / np.linalg.norm(perp), orth * np.linalg.norm(perp))):
        k = np.stack([key, np.zeros(d)])
        s = path_oracle_logits(q, k, w, b, 1, scale=1.0)
        assert abs(s[0] - expect) < 1e-13


# ------------------------------------------------------ I2: reflection = swap
def _read_swaps():
    cases = []
    with open(os.path.join(GOLDEN, "reflection_swap.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                head, x, y = line.split("|")
                d, a, bb = (int(t) for t in head.split())
                cases.append((d, a, bb, [float(t) for t in x.split()],
                              [float(t) for t in y.split()]))
    return cases


@pytest.mark.parametrize("d,a,bidx,x,y", _read_swaps())
def test_reflection_swaps_two_coordinates(d, a, bidx, x, y):
    wv = np.zeros(d)
    wv[a], wv[bidx] = 1 / math.sqrt(2), -1 / math.sqrt(2)
    q = np.stack([np.zeros(d), np.array(x)])
    w = np.stack([np.zeros(d), wv])
    b = np.array([0.0, 2.0])
    got = []
    for m in range(d):  # read z = H_1 q_1 coordinate by coordinate
        k = np.zeros((2, d))
        k[0, m] = 1.0
        got.append(path_oracle_logits(q, k, w, b, 1, scale=1.0)[0])
    np.testing.assert_allclose(got, y, atol=1e-14, rtol=0)


# ------------------------------------------------ I3: norms along the path
def _propagated(q, w, b, i):
    """z = H_1 ... H_i q_i read out with unit keys at position 0."""
    T, d = q.shape
    z = []
    for m in range(d):
        k = np.zeros((T, d))
        k[0, m] = 1.0
        z.append(path_oracle_logits(q, k, w, b, i, scale=1.0)[0])
    return np.array(z)


def test_reflections_preserve_norm_and_contractions_shrink():
    rng = np.random.default_rng(3)
    T, d = 30, 8
    q, _, _, w, b = _rand_inputs(rng, T, d)
    i = T - 1
    z2 = _propagated(q, w, np.full(T, 2.0), i)
    assert abs(np.linalg.norm(z2) - np.linalg.norm(q[i])) < 1e-12
    zb = _propagated(q, w, b, i)
    assert np.linalg.norm(zb) <= np.linalg.norm(q[i]) + 1e-12
    # beta = 2 carries an orthogonal map: z is not q itself (non-trivial path)
    assert np.linalg.norm(z2 - q[i]) > 1e-3


# --------------------------------------- I4: the linear-recurrence view
def test_logits_match_linear_recurrence():
    """S_t = S_{t-1} H_t + v_t k_t^T gives S_t q_t = sum_j v_j c_tj with
    c_tj = k_j^T H_{j+1}..H_t q_t (frame "PaTH keeps a recurrent path and a
    softmax readout")."""
    rng = np.random.default_rng(4)
    T, d = 25, 7
    q, k, v, w, b = _rand_inputs(rng, T, d)
    S = np.zeros((d, d))
    for t in range(T):
        Ht = np.eye(d) - b[t] * np.outer(w[t], w[t])
        S = S @ Ht + np.outer(v[t], k[t])
        c = path_oracle_logits(q, k, w, b, t, scale=1.0)
        np.testing.assert_allclose(S @ q[t], c @ v[: t + 1], atol=1e-11, rtol=0)


# ---------------------------------------------- I5: dense brute force
def test_logits_match_explicit_matrix_products():
    rng = np.random.default_rng(5)
    T, d = 18, 6
    q, k, _, w, b = _rand_inputs(rng, T, d)
    H = [np.eye(d) - b[t] * np.outer(w[t], w[t]) for t in range(T)]
    scale = 0.5
    for i in range(T):
        s = path_oracle_logits(q, k, w, b, i, scale=scale)
        for j in range(i + 1):
            P = np.eye(d)
            for t in range(j + 1, i + 1):  # H_{j+1} H_{j+2} ... H_i
                P = P @ H[t]
            assert abs(s[j] - scale * (k[j] @ P @ q[i])) < 1e-12


def test_product_order_matters():
    """Non-commuting transitions: the reversed order gives different logits,
    so the brute-force pin above is sensitive to orientation."""
    rng = np.random.default_rng(6)
    T, d = 6, 4
    q, k, _, w, b = _rand_inputs(rng, T, d)
    H = [np.eye(d) - b[t] * np.outer(w[t], w[t]) for t in range(T)]
    i, j = T - 1, 0
    fwd = np.eye(d)
    rev = np.eye(d)
    for t in range(j + 1, i + 1):
        fwd = fwd @ H[t]
        rev = H[t] @ rev
    s = path_oracle_logits(q, k, w, b, i, scale=1.0)[j]
    assert abs(s - k[j] @ fwd @ q[i]) < 1e-12
    assert abs(s - k[j] @ rev @ q[i]) > 1e-6


# ---------------------------------- I7: swap composition (golden closed form)
def _read_composition():
    ident_sum = other_max = None
    seqs = []
    with open(os.path.join(GOLDEN, "swap_composition.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("identity_sum"):
                ident_sum = int(line.split()[1])
            elif line.startswith("non_identity_max"):
                other_max = int(line.split()[1])
            else:
                kind, rest = line.split(":")
                pairs = [tuple(int(x) - 1 for x in m)
                         for m in re.findall(r"\((\d+),(\d+)\)", rest)]
                seqs.append((kind.strip(), pairs))
    return ident_sum, other_max, seqs


def test_swap_composition_score():
    ident_sum, other_max, seqs = _read_composition()
    assert ident_sum == 55 and other_max == 54
    d = 5
    ramp = np.arange(1, 6, dtype=np.float64)
    for kind, pairs in seqs:
        T = len(pairs) + 1
        q = np.zeros((T, d))
        q[-1] = ramp
        k = np.zeros((T, d))
        k[0] = ramp
        w = np.zeros((T, d))
        b = np.zeros(T)
        for t, (a, bb) in enumerate(pairs, start=1):
            w[t, a], w[t, bb] = 1 / math.sqrt(2), -1 / math.sqrt(2)
            b[t] = 2.0
        s = path_oracle_logits(q, k, w, b, T - 1, scale=1.0)[0]
        # the same permutation by moving labels (no linear algebra)
        lab = list(range(d))
        for a, bb in reversed(pairs):  # H_1 ... H_{T-1} q: H_{T-1} acts first
            lab[a], lab[bb] = lab[bb], lab[a]
        expect = float(sum((r + 1) * (lab[r] + 1) for r in range(d)))
        assert abs(s - expect) < 1e-12
        if kind == "identity":
            assert abs(s - ident_sum) < 1e-12
        else:
            assert s <= other_max + 1e-12


# ------------------------------------------------------------- I8: FoX gate
def test_fox_zero_gate_is_plain_path():
    rng = np.random.default_rng(8)
    T, d = 33, 8
    q, k, v, w, b = _rand_inputs(rng, T, d)
    o1, l1 = path_oracle_fwd(q, k, v, w, b)
    o2, l2 = path_oracle_fwd(q, k, v, w, b, logf=np.zeros(T))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_fox_constant_gate_with_beta_zero_is_linear_bias():
    """beta = 0 and log f = -c: log-weight = scale q_i.k_j - c (i - j); the
    gate sits outside the scaled logit (frame "FoX adds a separate mechanism
    for forgetting")."""
    rng = np.random.default_rng(9)
    T, d = 21, 5
    q, k, v, w, _ = _rand_inputs(rng, T, d)
    c, scale = 0.3, 0.7
    b = np.zeros(T)
    for i in (0, 7, T - 1):
        s = path_oracle_logits(q, k, w, b, i, logf=np.full(T, -c), scale=scale)
        expect = scale * (k[: i + 1] @ q[i]) - c * (i - np.arange(i + 1))
        np.testing.assert_allclose(s, expect, atol=1e-12, rtol=0)


def test_fox_gate_is_sum_over_open_interval():
    """The gate of (i, j) sums log f_s over s = j+1..i: f_j and earlier do not
    count, f_i does."""
    rng = np.random.default_rng(10)
    T, d = 9, 4
    q, k, _, w, b = _rand_inputs(rng, T, d)
    base = path_oracle_logits(q, k, w, b, T - 1)
    for s_idx in range(T):
        lf = np.zeros(T)
        lf[s_idx] = -1.0
        got = path_oracle_logits(q, k, w, b, T - 1, logf=lf)
        expect = base - np.array([1.0 if s_idx > j else 0.0 for j in range(T)])
        np.testing.assert_allclose(got, expect, atol=1e-13, rtol=0)


# --------------------------------------------------- softmax readout checks
def test_readout_invariants():
    rng = np.random.default_rng(11)
    T, d = 50, 8
    q, k, v, w, b = _rand_inputs(rng, T, d)
    ones = np.ones_like(v)
    out, lse = path_oracle_fwd(q, k, ones, w, b)
    np.testing.assert_allclose(out, 1.0, atol=1e-14, rtol=0)
    out, lse = path_oracle_fwd(q, k, v, w, b)
    for i in (0, 1, 25, T - 1):
        s = path_oracle_logits(q, k, w, b, i)
        assert s.max() - 1e-12 <= lse[i] <= s.max() + math.log(i + 1) + 1e-12
        p = np.exp(s - lse[i])
        assert abs(p.sum() - 1.0) < 1e-12
        np.testing.assert_allclose(out[i], p @ v[: i + 1], atol=1e-12, rtol=0)
    # row 0 attends only to itself
    np.testing.assert_allclose(out[0], v[0], atol=1e-15, rtol=0)


def test_row_sampling_matches_full_and_batching():
    rng = np.random.default_rng(12)
    B, H, T, d = 2, 3, 20, 4
    x = [rng.standard_normal((B, H, T, d)) for _ in range(4)]
    w = x[3] / np.linalg.norm(x[3], axis=-1, keepdims=True)
    b = 2.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T))))
    lf = -np.abs(rng.standard_normal((B, H, T))) * 0.1
    out, lse = path_oracle_fwd(x[0], x[1], x[2], w, b, logf=lf, threads=3)
    rows = [0, 5, 19, 20, 41, B * H * T - 1]
    o2, l2 = path_oracle_fwd(x[0], x[1], x[2], w, b, logf=lf, rows=rows, threads=2)
    np.testing.assert_array_equal(o2, out.reshape(-1, d)[rows])
    np.testing.assert_array_equal(l2, lse.reshape(-1)[rows])
    # each (b, h) is an independent problem
    o3, l3 = path_oracle_fwd(x[0][1, 2], x[1][1, 2], x[2][1, 2], w[1, 2], b[1, 2],
                             logf=lf[1, 2])
    np.testing.assert_array_equal(o3, out[1, 2])
    np.testing.assert_array_equal(l3, lse[1, 2])


def test_oracle_rejects_bad_rows():
    rng = np.random.default_rng(13)
    q, k, v, w, b = _rand_inputs(rng, 5, 3)
    with pytest.raises(RuntimeError):
        path_oracle_fwd(q, k, v, w, b, rows=[5])


# ------------------------------------------- decoding: keys rewritten in place
def test_decoded_keys_give_the_path_logits():
    """(k_j^(t))^T q_t = k_j^T H_{j+1} .. H_t q_t (frame "Decoding updates
    historical keys in place"), checked against the pinned logits."""
    rng = np.random.default_rng(21)
    T, d = 26, 7
    q, k, _, w, b = _rand_inputs(rng, T, d)
    for t in (0, 1, 12, T - 1):
        kt = path_oracle_decoded_keys(k, w, b, t)
        s = path_oracle_logits(q, k, w, b, t, scale=1.0)
        np.testing.assert_allclose(kt @ q[t], s, atol=1e-12, rtol=0)
        np.testing.assert_array_equal(kt[t], k[t])  # the newest key is untouched


def test_decoded_keys_match_explicit_products_and_one_step_update():
    rng = np.random.default_rng(22)
    T, d = 12, 5
    _, k, _, w, b = _rand_inputs(rng, T, d)
    H = [np.eye(d) - b[t] * np.outer(w[t], w[t]) for t in range(T)]
    t = T - 1
    kt = path_oracle_decoded_keys(k, w, b, t)
    for j in range(t + 1):
        P = np.eye(d)
        for s_ in range(j + 1, t + 1):  # H_t ... H_{j+1}
            P = H[s_] @ P
        np.testing.assert_allclose(kt[j], P @ k[j], atol=1e-12)
    # one decoding step is the rank-one rewrite of every earlier key
    prev = path_oracle_decoded_keys(k, w, b, t - 1)
    step = prev - b[t] * np.outer(prev @ w[t], w[t])
    np.testing.assert_allclose(kt[:t], step, atol=1e-12)


@pytest.mark.parametrize("fox", [False, True])
def test_decoding_token_by_token_reproduces_the_forward(fox):
    """Decoding from an empty cache gives every row of the (pinned) forward,
    and leaves the cache holding the keys aligned to the last token."""
    rng = np.random.default_rng(23)
    T, d = 33, 6
    q, k, v, w, b = _rand_inputs(rng, T, d)
    logf = np.log(rng.uniform(0.6, 1.0, T)) if fox else None
    scale = 0.41
    ref_out, ref_lse = path_oracle_fwd(q, k, v, w, b, logf=logf, scale=scale)
    kc, vc = np.zeros((T, d)), np.zeros((T, d))
    lam = np.zeros(T) if fox else None
    for t in range(T):
        o, l = path_oracle_decode_step(kc, vc, lam, q[t], k[t], v[t], w[t], b[t],
                                       None if logf is None else logf[t], t, scale=scale)
        np.testing.assert_allclose(o, ref_out[t], atol=1e-12, rtol=0)
        assert abs(l - ref_lse[t]) < 1e-12
    np.testing.assert_allclose(kc, path_oracle_decoded_keys(k, w, b, T - 1), atol=1e-12)
    np.testing.assert_array_equal(vc, v)
    if fox:
        np.testing.assert_allclose(lam, np.cumsum(logf), atol=1e-13)


def test_decoding_first_token_attends_to_itself():
    rng = np.random.default_rng(24)
    d = 5
    q, k, v, w, b = _rand_inputs(rng, 1, d)
    kc, vc = np.zeros((1, d)), np.zeros((1, d))
    o, l = path_oracle_decode_step(kc, vc, None, q[0], k[0], v[0], w[0], b[0], None, 0,
                                   scale=0.3)
    np.testing.assert_array_equal(o, v[0])
    assert abs(l - 0.3 * (k[0] @ q[0])) < 1e-15


# --------------------------------------------------------------- partial PaTH
def test_partial_path_full_width_is_path_and_zero_width_is_plain_attention():
    rng = np.random.default_rng(25)
    T, d = 30, 8
    q, k, v, w, b = _rand_inputs(rng, T, d)
    logf = np.log(rng.uniform(0.7, 1.0, T))
    o1, l1 = path_oracle_partial_fwd(q, k, v, w, b, logf=logf, scale=0.4)
    o2, l2 = path_oracle_fwd(q, k, v, w, b, logf=logf, scale=0.4)
    np.testing.assert_allclose(o1, o2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-13, rtol=0)
    o0, l0 = path_oracle_partial_fwd(q, k, v, np.zeros((T, 0)), b, scale=0.4)
    ref_out, ref_lse = _causal_softmax_attention(q, k, v, 0.4)
    np.testing.assert_allclose(o0, ref_out, atol=1e-13, rtol=0)
    np.testing.assert_allclose(l0, ref_lse, atol=1e-13, rtol=0)


def test_partial_path_matches_block_diagonal_transitions():
    """Brute force: H_t = blockdiag(I_r - beta u u^T, I_{d-r}) as explicit
    matrices, and the same logits from full PaTH with u zero-padded to d."""
    rng = np.random.default_rng(26)
    T, d, r = 14, 7, 3
    q, k, v, _, b = _rand_inputs(rng, T, d)
    u = rng.standard_normal((T, r))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    scale = 0.6
    out, lse = path_oracle_partial_fwd(q, k, v, u, b, scale=scale)
    H = []
    for t in range(T):
        M = np.eye(d)
        M[:r, :r] -= b[t] * np.outer(u[t], u[t])
        H.append(M)
    for i in range(T):
        s = np.zeros(i + 1)
        for j in range(i + 1):
            P = np.eye(d)
            for t in range(j + 1, i + 1):
                P = P @ H[t]
            s[j] = scale * (k[j] @ P @ q[i])
        p = np.exp(s - s.max())
        np.testing.assert_allclose(out[i], p @ v[: i + 1] / p.sum(), atol=1e-12)
        assert abs(lse[i] - (s.max() + np.log(p.sum()))) < 1e-12
    wpad = np.concatenate([u, np.zeros((T, d - r))], axis=1)
    o2, _ = path_oracle_fwd(q, k, v, wpad, b, scale=scale)
    np.testing.assert_allclose(out, o2, atol=1e-12)
