"""Checks that pin the float64 oracle to what the pages and mathematics fix.

Each ``check_*`` takes an oracle ``mha`` callable (signature of
``oracle.Oracle.mha``) and raises AssertionError when the oracle disagrees.
They are run on the real oracle (test_oracle_pins.py) and on deliberately
broken builds of it (test_oracle_mutants.py), where at least one must fail.

Nothing here re-types the oracle's loop: expected values come from the pages'
printed numbers (``tests/golden``), closed forms, a different algebraic form
of the same weights (the temperature form), pure-Python brute force with
``math.fsum`` and no max-subtraction, or torch's CPU float64 SDPA.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

NONE, CAUSAL, KEYPAD = 0, 1, 2


def _golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _weights(mha, q_vec, keys, scale=None):
    """Weights of one query over n keys, read through one-hot value rows.

    With value row j = e_j (d >= n) the output is the weight vector itself.
    Keys and query are zero-padded to d = max(n, len(q)); padding adds 0 to
    every dot product, so with an explicit scale nothing else changes.
    """
    keys = np.asarray(keys, dtype=np.float64)
    n, dk = keys.shape
    d = max(n, dk)
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, :dk] = q_vec
    k = np.zeros((1, n, 1, d))
    k[0, :, 0, :dk] = keys
    v = np.zeros((1, n, 1, d))
    v[0, np.arange(n), 0, np.arange(n)] = 1.0
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    o = mha(q, k, v, scale=scale)
    return o[0, 0, 0, :n]


# --------------------------------------------------------------------------
# the pages' worked examples
# --------------------------------------------------------------------------
def check_worked_example(mha):
    """Formula page, 応用: 8 words, d_k = 4, query of それ."""
    g = _golden("cat_fish_worked_example.json")
    keys = np.array(g["keys"], dtype=np.float64)
    words = g["words"]
    q = np.array(g["query"], dtype=np.float64)
    p = g["printed"]
    # output with values = keys and the default scale 1/sqrt(4) (the page divides by 2)
    o, lse = mha(q.reshape(1, 1, 1, 4), keys.reshape(1, 8, 1, 4),
                 keys.reshape(1, 8, 1, 4), return_lse=True)
    assert np.allclose(o.ravel(), p["output"], atol=0.006), o.ravel()
    assert abs(math.exp(lse.ravel()[0]) - p["sum_of_exponentials"]) < 0.01
    a = _weights(mha, q, keys, scale=0.5)
    w = {words[j]: a[j] for j in range(8)}
    for word in ("魚", "おいしかった", "それ"):
        assert abs(w[word] - p["weights"][word]) < 0.0006, (word, w[word])
    for word in ("ねこ", "が", "を", "食べた", "は"):
        assert abs(w[word] - p["weights"]["others"]) < 0.0006, (word, w[word])
    # not divided (scale 1) and divided by 8 (scale 1/8)
    a1 = _weights(mha, q, keys, scale=1.0)
    assert abs(a1[words.index("魚")] - p["fish_weight_scale_1"]) < 0.0006
    a8 = _weights(mha, q, keys, scale=1.0 / 8.0)
    assert abs(a8[words.index("魚")] - p["fish_weight_scale_1_over_8"]) < 0.0006


def check_two_key_example(mha):
    """Formula page, 応用 (次元が 64 なら): d_k = 64, dot products 8 apart."""
    g = _golden("two_key_d64.json")
    p = g["printed"]
    rng = _rng(7)
    q = rng.standard_normal(64)
    k1 = rng.standard_normal(64)
    k2 = k1 - g["dot_product_gap"] * q / (q @ q)  # q.k1 - q.k2 = 8
    keys = np.stack([k1, k2])
    # unscaled (Luong) attention
    a = _weights(mha, q, keys, scale=1.0)
    assert abs(a[0] - p["unscaled_weights"][0]) < 5e-5
    assert abs(a[1] - p["unscaled_weights"][1]) < 5e-5
    assert abs(a[0] / a[1] - p["unscaled_ratio"]) / p["unscaled_ratio"] < 1e-3
    g_unscaled = a[0] * (1 - a[0])
    assert abs(g_unscaled - p["unscaled_a_one_minus_a"]) < 5e-5
    # default scale must be 1/sqrt(64) = 1/8: weights 0.731 / 0.269
    qd = q.reshape(1, 1, 1, 64)
    kd = keys.reshape(1, 2, 1, 64)
    vd = np.zeros((1, 2, 1, 64))
    vd[0, 0, 0, 0] = 1.0
    vd[0, 1, 0, 1] = 1.0
    o = mha(qd, kd, vd)  # scale left to its default
    a = o[0, 0, 0, :2]
    assert abs(a[0] - p["scaled_weights"][0]) < 5e-4, a
    assert abs(a[1] - p["scaled_weights"][1]) < 5e-4, a
    assert abs(a[0] / a[1] - p["scaled_ratio"]) < 5e-3
    g_scaled = a[0] * (1 - a[0])
    assert abs(g_scaled - p["scaled_a_one_minus_a"]) < 5e-4
    assert abs(g_scaled / g_unscaled - p["gradient_gain"]) < 10


def check_toy_shape(mha):
    """Cookipedia toy model: d_model 6, 2 heads, target 4, source 8 -> [1, 4, 6]."""
    rng = _rng(11)
    q = rng.standard_normal((1, 4, 2, 3))
    k = rng.standard_normal((1, 8, 2, 3))
    v = rng.standard_normal((1, 8, 2, 3))
    o = mha(q, k, v)
    assert o.shape == (1, 4, 2, 3)
    assert o.reshape(1, 4, 6).shape == (1, 4, 6)
    # each head attends only within its own slice of the 6-dim vector
    o_h0 = mha(q[:, :, :1], k[:, :, :1], v[:, :, :1])
    assert np.array_equal(o[:, :, :1], o_h0)


# --------------------------------------------------------------------------
# closed forms and invariants (formula page, 証明 and 応用)
# --------------------------------------------------------------------------
def check_weights_positive_sum_one(mha):
    rng = _rng(1)
    for n in (1, 2, 7, 16):
        q = rng.standard_normal(16)
        keys = rng.standard_normal((n, 16))
        a = _weights(mha, q, keys)
        assert np.all(a > 0)
        assert abs(a.sum() - 1.0) < 1e-13


def check_shift_invariance(mha):
    """Adding one constant to every score leaves the weights unchanged."""
    rng = _rng(2)
    B, L, H, d = 2, 9, 3, 8
    q = rng.standard_normal((B, L, H, d))
    k = rng.standard_normal((B, L, H, d))
    v = rng.standard_normal((B, L, H, d))
    scale = 0.3
    o = mha(q, k, v, scale=scale)
    for c in (-40.0, 3.5, 250.0):
        # extra component: q gets 1, every key gets c/scale -> score + c
        q2 = np.concatenate([q, np.ones((B, L, H, 1))], axis=-1)
        k2 = np.concatenate([k, np.full((B, L, H, 1), c / scale)], axis=-1)
        v2 = np.concatenate([v, np.zeros((B, L, H, 1))], axis=-1)
        o2 = mha(q2, k2, v2, scale=scale)
        assert np.allclose(o2[..., :d], o, rtol=0, atol=1e-12)


def check_weight_ratio(mha):
    """a_j / a_i = e^{s_j - s_i}, scores from numpy's dot."""
    rng = _rng(3)
    q = rng.standard_normal(12)
    keys = rng.standard_normal((10, 12))
    scale = 0.4
    a = _weights(mha, q, keys, scale=scale)
    s = scale * (keys @ q)
    for i in range(10):
        for j in range(10):
            assert abs(a[j] / a[i] - math.exp(s[j] - s[i])) <= 1e-12 * math.exp(s[j] - s[i])


def check_temperature_form(mha):
    """a_j = 1 / sum_i e^{(z_i - z_j)/tau} with z = q.k and tau = 1/scale."""
    rng = _rng(4)
    q = rng.standard_normal(8)
    keys = rng.standard_normal((6, 8))
    z = keys @ q
    for tau in (0.25, 1.0, math.sqrt(8), 10.0):
        a = _weights(mha, q, keys, scale=1.0 / tau)
        ref = np.array([1.0 / sum(math.exp((z[i] - z[j]) / tau) for i in range(6))
                        for j in range(6)])
        assert np.allclose(a, ref, rtol=1e-12, atol=0)


def check_limits(mha):
    """tau -> 0 selects the argmax value row; tau -> inf gives the plain mean."""
    rng = _rng(5)
    B, Lq, Lk, H, d = 1, 4, 11, 2, 6
    q = rng.standard_normal((B, Lq, H, d))
    k = rng.standard_normal((B, Lk, H, d))
    v = rng.standard_normal((B, Lk, H, d))
    z = np.einsum("bihd,bjhd->bhij", q, k)
    o_cold = mha(q, k, v, scale=1e6)
    o_hot = mha(q, k, v, scale=1e-30)
    for h in range(H):
        for i in range(Lq):
            j = int(np.argmax(z[0, h, i]))
            assert np.array_equal(o_cold[0, i, h], v[0, j, h])
            assert np.allclose(o_hot[0, i, h], v[0, :, h].mean(axis=0), rtol=0, atol=1e-14)
    # equal scores (identical keys) give the mean of the value rows at any scale
    k_same = np.repeat(k[:, :1], Lk, axis=1)
    o_eq = mha(q, k_same, v, scale=2.0)
    assert np.allclose(o_eq[0], np.broadcast_to(v[0].mean(axis=0), (Lq, H, d)),
                       rtol=0, atol=1e-14)
    # tied maxima share the weight equally (mean of the tied rows as tau -> 0)
    k_tie = k.copy()
    k_tie[0, 3] = k_tie[0, 7]
    z = np.einsum("bihd,bjhd->bhij", q, k_tie)
    o_cold = mha(q, k_tie, v, scale=1e6)
    for h in range(H):
        for i in range(Lq):
            if int(np.argmax(z[0, h, i])) in (3, 7):
                want = 0.5 * (v[0, 3, h] + v[0, 7, h])
                assert np.allclose(o_cold[0, i, h], want, rtol=0, atol=1e-14)


def check_lse_bounds(mha):
    """max s <= log sum e^s <= max s + log n (formula page, 広がる学問, 数学)."""
    rng = _rng(6)
    B, L, H, d = 2, 13, 2, 5
    q = rng.standard_normal((B, L, H, d)) * 3
    k = rng.standard_normal((B, L, H, d)) * 3
    v = rng.standard_normal((B, L, H, d))
    _, lse = mha(q, k, v, return_lse=True)
    s = np.einsum("bihd,bjhd->bhij", q, k) / math.sqrt(d)
    mx = s.max(axis=-1)
    assert np.all(mx <= lse + 1e-12)
    assert np.all(lse <= mx + math.log(L) + 1e-12)
    assert np.allclose(lse, np.log(np.exp(s).sum(axis=-1)), rtol=1e-13, atol=1e-12)


# --------------------------------------------------------------------------
# masks (cookipedia decoder section; formula page 応用, 先を読まない仕掛け)
# --------------------------------------------------------------------------
def check_causal(mha):
    rng = _rng(8)
    B, L, H, d = 2, 10, 3, 4
    q = rng.standard_normal((B, L, H, d))
    k = rng.standard_normal((B, L, H, d))
    v = rng.standard_normal((B, L, H, d))
    o = mha(q, k, v, CAUSAL)
    for t in range(L):
        # keys after t do not influence rows <= t (bit-identical)
        k2 = k.copy()
        v2 = v.copy()
        k2[:, t + 1:] = rng.standard_normal(k2[:, t + 1:].shape) * 5
        v2[:, t + 1:] = rng.standard_normal(v2[:, t + 1:].shape) * 5
        o2 = mha(q, k2, v2, CAUSAL)
        assert np.array_equal(o2[:, :t + 1], o[:, :t + 1])
        # row t equals unmasked attention of query t over keys 0..t
        ot = mha(q[:, t:t + 1], k[:, :t + 1], v[:, :t + 1])
        assert np.array_equal(ot[:, 0], o[:, t])
    # the diagonal is kept: row 0 sees exactly key 0
    assert np.array_equal(o[:, 0], v[:, 0])
    # masked weights are exactly 0, the rest sum to 1
    qd = rng.standard_normal((1, 6, 1, 6))
    kd = rng.standard_normal((1, 6, 1, 6))
    vd = np.eye(6).reshape(1, 6, 1, 6)
    a = mha(qd, kd, vd, CAUSAL, scale=0.7)[0, :, 0, :]
    for i in range(6):
        assert np.all(a[i, i + 1:] == 0.0)
        assert np.all(a[i, :i + 1] > 0.0)
        assert abs(a[i].sum() - 1.0) < 1e-14


def check_key_padding(mha):
    rng = _rng(9)
    B, Lq, Lk, H, d = 4, 5, 9, 2, 9
    q = rng.standard_normal((B, Lq, H, d))
    k = rng.standard_normal((B, Lk, H, d))
    v = rng.standard_normal((B, Lk, H, d))
    lens = np.array([9, 1, 4, 7], dtype=np.int32)
    o = mha(q, k, v, KEYPAD, key_lens=lens)
    for b in range(B):
        n = int(lens[b])
        # equals unmasked attention over the first n keys (bit-identical)
        ob = mha(q[b:b + 1], k[b:b + 1, :n], v[b:b + 1, :n])
        assert np.array_equal(ob[0], o[b])
    # keys past the length do not matter at all
    k2 = k.copy()
    v2 = v.copy()
    for b in range(B):
        k2[b, lens[b]:] = 1e3
        v2[b, lens[b]:] = -7.0
    assert np.array_equal(mha(q, k2, v2, KEYPAD, key_lens=lens), o)
    # weights of padded keys are exactly 0
    vd = np.zeros((B, Lk, H, d))
    for j in range(Lk):
        vd[:, j, :, j] = 1.0
    a = mha(q, k, vd, KEYPAD, key_lens=lens)
    for b in range(B):
        assert np.all(a[b, :, :, lens[b]:] == 0.0)
        assert np.allclose(a[b].sum(axis=-1), 1.0, rtol=0, atol=1e-14)
    # lengths outside [0, Lk] clamp; a row with no key gives 0
    lens2 = np.array([0, 100, -3, 9], dtype=np.int32)
    o2, lse2 = mha(q, k, v, KEYPAD, key_lens=lens2, return_lse=True)
    assert np.all(o2[0] == 0.0) and np.all(o2[2] == 0.0)
    assert np.all(np.isneginf(lse2[0])) and np.all(np.isneginf(lse2[2]))
    assert np.array_equal(o2[1], mha(q[1:2], k[1:2], v[1:2])[0])


def check_combined_mask(mha):
    """Both masks (kind 3): row i of sequence b sees keys j <= i with
    j < key_lens[b].  Rows below the length equal the causal rows and rows at or
    past it equal the key-padding rows, bit for bit; keys a row may not see do
    not matter at all."""
    rng = _rng(14)
    B, L, H, d = 4, 9, 2, 5
    q = rng.standard_normal((B, L, H, d))
    k = rng.standard_normal((B, L, H, d))
    v = rng.standard_normal((B, L, H, d))
    lens = np.array([9, 3, 0, 6], dtype=np.int32)
    o, lse = mha(q, k, v, CAUSAL | KEYPAD, key_lens=lens, return_lse=True)
    oc = mha(q, k, v, CAUSAL)
    op = mha(q, k, v, KEYPAD, key_lens=lens)
    for b in range(B):
        n = int(lens[b])
        assert np.array_equal(o[b, :n], oc[b, :n])
        assert np.array_equal(o[b, n:], op[b, n:])
    # sequence 2 has no key: every row is 0 with log-sum-exp -inf
    assert np.all(o[2] == 0.0) and np.all(np.isneginf(lse[2]))
    # perturbing every key a row may not see changes nothing
    for b in range(B):
        for i in range(L):
            n_vis = min(i + 1, int(lens[b]))
            k2 = k.copy()
            v2 = v.copy()
            k2[b, n_vis:] = rng.standard_normal(k2[b, n_vis:].shape) * 7
            v2[b, n_vis:] = rng.standard_normal(v2[b, n_vis:].shape) * 7
            o2 = mha(q, k2, v2, CAUSAL | KEYPAD, key_lens=lens)
            assert np.array_equal(o2[b, i], o[b, i])
    # removed weights are exactly 0, the rest sum to 1
    vd = np.zeros((B, L, H, L))
    for j in range(L):
        vd[:, j, :, j] = 1.0
    a = mha(q, k, vd, CAUSAL | KEYPAD, key_lens=lens)
    for b in range(B):
        for i in range(L):
            n_vis = min(i + 1, int(lens[b]))
            assert np.all(a[b, i, :, n_vis:] == 0.0)
            if n_vis > 0:
                assert np.all(a[b, i, :, :n_vis] > 0.0)
                assert np.allclose(a[b, i].sum(axis=-1), 1.0, rtol=0, atol=1e-14)


def check_value_width(mha):
    """d_v != d_k (Equation (1) takes values of width d_v): every output column
    is the same weighted mean of one value column, so splitting the value
    columns splits the output columns bit for bit, and the weights (read off
    with one-hot values, d_v = Lk) do not depend on d_v."""
    rng = _rng(15)
    B, Lq, Lk, H, d = 2, 6, 7, 3, 4
    q = rng.standard_normal((B, Lq, H, d))
    k = rng.standard_normal((B, Lk, H, d))
    v = rng.standard_normal((B, Lk, H, 11))
    for mask, lens in ((NONE, None), (KEYPAD, np.array([7, 2], dtype=np.int32))):
        o = mha(q, k, v, mask, key_lens=lens)
        assert o.shape == (B, Lq, H, 11)
        o1 = mha(q, k, np.ascontiguousarray(v[..., :5]), mask, key_lens=lens)
        o2 = mha(q, k, np.ascontiguousarray(v[..., 5:]), mask, key_lens=lens)
        assert np.array_equal(o[..., :5], o1) and np.array_equal(o[..., 5:], o2)
        for c in range(11):
            oc = mha(q, k, np.ascontiguousarray(v[..., c:c + 1]), mask, key_lens=lens)
            assert np.array_equal(o[..., c:c + 1], oc)
    # the scale defaults to 1/sqrt(d_k), not 1/sqrt(d_v)
    onehot = np.zeros((B, Lk, H, Lk))
    for j in range(Lk):
        onehot[:, j, :, j] = 1.0
    a = mha(q, k, onehot)
    a_ref = mha(q, k, onehot, scale=1.0 / math.sqrt(d))
    assert np.array_equal(a, a_ref)
    s = np.einsum("bihc,bjhc->bihj", q, k) / math.sqrt(d)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    assert np.allclose(a, e / e.sum(axis=-1, keepdims=True), rtol=0, atol=1e-14)


def check_empty(mha):
    rng = _rng(10)
    q = rng.standard_normal((2, 3, 2, 4))
    o = mha(q, np.zeros((2, 0, 2, 4)), np.zeros((2, 0, 2, 4)))
    assert o.shape == (2, 3, 2, 4) and np.all(o == 0.0)
    o = mha(np.zeros((0, 3, 2, 4)), np.zeros((0, 5, 2, 4)), np.zeros((0, 5, 2, 4)))
    assert o.shape == (0, 3, 2, 4)


# --------------------------------------------------------------------------
# brute force and a library cross-check
# --------------------------------------------------------------------------
def brute_force(q, k, v, mask_kind=NONE, key_lens=None, scale=None):
    """Pure Python with math.fsum: weights e^{s_j} / sum e^{s_i} exactly as
    written, no max-subtraction (inputs kept small so nothing overflows).
    The value width d_v (v's last axis) may differ from d_k; mask kind 3
    keeps key j for row i only when j <= i and j < key_lens[b]."""
    B, Lq, H, d = q.shape
    Lk = k.shape[1]
    d_v = v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, Lq, H, d_v))
    for b in range(B):
        for h in range(H):
            for i in range(Lq):
                keys = [j for j in range(Lk)
                        if not (mask_kind & CAUSAL and j > i)
                        and not (mask_kind & KEYPAD and j >= int(key_lens[b]))]
                if not keys:
                    continue
                e = {j: math.exp(scale * math.fsum(float(q[b, i, h, c]) * float(k[b, j, h, c])
                                                   for c in range(d))) for j in keys}
                total = math.fsum(e.values())
                for c in range(d_v):
                    out[b, i, h, c] = math.fsum(e[j] / total * float(v[b, j, h, c]) for j in keys)
    return out


def check_brute_force(mha):
    rng = _rng(12)
    for trial in range(16):
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 3))
        d = int(rng.integers(1, 5))
        # every third trial a wider value row (d_v > d_k)
        d_v = d + int(rng.integers(1, 4)) if trial % 3 == 2 else d
        Lk = int(rng.integers(1, 6))
        mask = trial % 4
        Lq = Lk if mask & CAUSAL else int(rng.integers(1, 6))
        q = rng.standard_normal((B, Lq, H, d))
        k = rng.standard_normal((B, Lk, H, d))
        v = rng.standard_normal((B, Lk, H, d_v))
        lens = rng.integers(0, Lk + 1, size=B).astype(np.int32) if mask & KEYPAD else None
        scale = None if trial % 2 == 0 else float(rng.uniform(0.1, 2.0))
        o = mha(q, k, v, mask, key_lens=lens, scale=scale)
        ref = brute_force(q, k, v, mask, lens, scale)
        assert np.allclose(o, ref, rtol=0, atol=1e-12), (trial, np.abs(o - ref).max())


def check_torch_sdpa(mha):
    """torch's CPU float64 scaled_dot_product_attention with an explicit mask."""
    import torch
    import torch.nn.functional as F
    rng = _rng(13)
    for mask, d_v in ((NONE, 16), (CAUSAL, 16), (KEYPAD, 16), (CAUSAL | KEYPAD, 16),
                      (NONE, 24), (CAUSAL | KEYPAD, 40)):
        B, H, d = 3, 4, 16
        Lq, Lk = (41, 41) if mask & CAUSAL else (29, 41)
        q = rng.standard_normal((B, Lq, H, d))
        k = rng.standard_normal((B, Lk, H, d))
        v = rng.standard_normal((B, Lk, H, d_v))
        lens = np.array([41, 1, 17], dtype=np.int32) if mask & KEYPAD else None
        o = mha(q, k, v, mask, key_lens=lens)
        allowed = torch.ones(B, 1, Lq, Lk, dtype=torch.bool)
        if mask & CAUSAL:
            allowed &= torch.ones(Lq, Lk, dtype=torch.bool).tril()
        if mask & KEYPAD:
            for b in range(B):
                allowed[b, :, :, int(lens[b]):] = False
        # every row keeps at least key 0 (torch's softmax of an empty row is NaN)
        assert allowed.any(dim=-1).all()
        tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=allowed)
        ref = ref.permute(0, 2, 1, 3).numpy()
        assert np.allclose(o, ref, rtol=0, atol=1e-12), (mask, np.abs(o - ref).max())


ALL_CHECKS = [
    check_worked_example, check_two_key_example, check_toy_shape,
    check_weights_positive_sum_one, check_shift_invariance, check_weight_ratio,
    check_temperature_form, check_limits, check_lse_bounds, check_causal,
    check_key_padding, check_combined_mask, check_value_width, check_empty, check_brute_force,
    check_torch_sdpa,
]
