"""Pins of the oracle's gradient (oracle.mha_bwd), independent of its code.

Each check takes ``mha`` (the forward, oracle.mha's signature) and ``bwd``
(the gradient, oracle.mha_bwd's signature):

  - finite differences: the gradient of L = sum(dout * O) with respect to every
    element of q, k and v, by central differences of the FORWARD oracle, on
    tiny cases of every mask and an explicit scale;
  - torch: float64 autograd of an explicitly written masked softmax attention;
  - invariants: the weights of a row sum to 1, so sum_j dL/ds_j = 0 and hence
    sum_j dk_j = 0 for every head; sum_j dv_j = sum of dout over rows that see
    a key; removed keys get exactly zero gradient; a row that sees one key has
    dq = 0 exactly (its weight is 1 whatever the score); q = 0 gives dk = 0;
    the gradient is linear in dout.
"""
from __future__ import annotations

import numpy as np

NONE, CAUSAL, KEYPAD = 0, 1, 2


def _case(seed, B, Lq, H, Lk, d):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, Lq, H, d))
    k = r.standard_normal((B, Lk, H, d))
    v = r.standard_normal((B, Lk, H, d))
    dout = r.standard_normal((B, Lq, H, d))
    return q, k, v, dout


def check_bwd_finite_differences(mha, bwd):
    cases = [((1, 3, 2, 3, 3), NONE, None, None),
             ((2, 4, 1, 4, 3), CAUSAL, None, 0.7),
             ((2, 3, 2, 5, 2), KEYPAD, [5, 2], None),
             ((2, 4, 1, 4, 2), CAUSAL | KEYPAD, [4, 2], None)]
    h = 1e-6
    for seed, (shape, mask, lens, scale) in enumerate(cases):
        q, k, v, dout = _case(100 + seed, *shape)
        grads = bwd(q, k, v, dout, mask, key_lens=lens, scale=scale)

        def loss(qq, kk, vv):
            return float(np.sum(dout * mha(qq, kk, vv, mask, key_lens=lens, scale=scale)))

        for which, g in zip(range(3), grads):
            x = [q, k, v][which]
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][idx] += h
                args_m[which][idx] -= h
                fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
                assert abs(fd - g[idx]) <= 1e-7 * (1 + abs(fd)), \
                    (shape, mask, which, idx, fd, g[idx])


def check_bwd_torch_autograd(mha, bwd):
    import torch
    for seed, (shape, mask, lens) in enumerate([((2, 9, 3, 11, 5), NONE, None),
                                                ((2, 10, 2, 10, 4), CAUSAL, None),
                                                ((3, 7, 2, 12, 6), KEYPAD, [12, 1, 5]),
                                                ((3, 8, 2, 8, 4), CAUSAL | KEYPAD, [8, 1, 5])]):
        q, k, v, dout = _case(200 + seed, *shape)
        B, Lq, H, Lk, d = shape
        scale = 1.0 / np.sqrt(d)
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        s = torch.einsum("bihd,bjhd->bhij", tq, tk) * scale
        keep = torch.ones(B, 1, Lq, Lk, dtype=torch.bool)
        if mask & CAUSAL:
            keep = keep & torch.tril(torch.ones(Lq, Lk, dtype=torch.bool))
        if mask & KEYPAD:
            for b, n in enumerate(lens):
                keep[b, :, :, n:] = False
        s = s.masked_fill(~keep, float("-inf"))
        o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), tv)
        o.backward(torch.tensor(dout))
        got = bwd(q, k, v, dout, mask, key_lens=lens)
        for t, g in zip((tq, tk, tv), got):
            assert np.allclose(g, t.grad.numpy(), rtol=1e-10, atol=1e-12)


def check_bwd_invariants(mha, bwd):
    q, k, v, dout = _case(300, 2, 6, 3, 9, 4)
    lens = [9, 4]
    dq, dk, dv = bwd(q, k, v, dout, KEYPAD, key_lens=lens)
    for b, n in enumerate(lens):
        assert np.allclose(dk[b].sum(axis=0), 0.0, atol=1e-12)          # sum_j dk_j = 0
        assert np.allclose(dv[b].sum(axis=0), dout[b].sum(axis=0), atol=1e-12)
        assert np.all(dk[b, n:] == 0.0) and np.all(dv[b, n:] == 0.0)   # removed keys
    # causal: row 0 sees one key, so its weight is 1 whatever the score
    q, k, v, dout = _case(301, 2, 7, 2, 7, 3)
    dq, dk, dv = bwd(q, k, v, dout, CAUSAL)
    assert np.all(dq[:, 0] == 0.0)
    assert np.allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    # keys past the last query get nothing under the causal mask only through
    # later rows: the last key is seen by the last row alone, with weight a
    assert not np.all(dv[:, -1] == 0.0)
    # q = 0: every score 0, weights uniform, and dk = scale * ds * q = 0
    dq0, dk0, dv0 = bwd(np.zeros_like(q), k, v, dout, NONE)
    assert np.all(dk0 == 0.0)
    n = k.shape[1]
    assert np.allclose(dv0, np.broadcast_to(dout.sum(axis=1, keepdims=True) / n, dv0.shape),
                       atol=1e-12)
    # linear in dout
    a = bwd(q, k, v, dout, NONE)
    b2 = bwd(q, k, v, 2.0 * dout, NONE)
    for x, y in zip(a, b2):
        assert np.allclose(2.0 * x, y, rtol=1e-12, atol=1e-14)


ALL_BWD_CHECKS = [check_bwd_finite_differences, check_bwd_torch_autograd, check_bwd_invariants]
