"""The oracle's multi-head layer (oracle.mha_layer) against what fixes it
independently (CPU only):

  - torch's float64 nn.MultiheadAttention with the biases off, whose weight
    layout is its own ([3E, E] applied as x W^T), self- and cross-attention,
    every mask;
  - identity weights (d_model = H d_k): the layer reduces to the attention of
    the heads of x, which the attention pins fix;
  - Section 3.2.2 written head by head in plain numpy (its own softmax, no C
    oracle): head_h = softmax(X W_h^Q (M W_h^K)^T / sqrt(d_k)) M W_h^V, then
    Concat(head_1 .. head_H) W^O;
and planted mistakes in copies of the layer (on the CPU) each fail one of them.
"""
import math

import numpy as np
import pytest

import oracle

NONE, CAUSAL, KEYPAD, BOTH = 0, 1, 2, 3


def _case(seed, B, Lq, Lk, d_model, H, d_k, cross):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, Lq, d_model))
    mem = rng.standard_normal((B, Lk, d_model)) if cross else None
    w_qkv = rng.standard_normal((d_model, 3 * H * d_k)) / math.sqrt(d_model)
    w_o = rng.standard_normal((H * d_k, d_model)) / math.sqrt(H * d_k)
    return x, mem, w_qkv, w_o


def per_head_numpy(x, w_qkv, w_o, H, mem=None, mask_kind=NONE, key_lens=None):
    """Section 3.2.2 head by head, numpy only."""
    mem = x if mem is None else mem
    B, Lq, _ = x.shape
    Lk = mem.shape[1]
    hd = w_qkv.shape[1] // 3
    d_k = hd // H
    heads = []
    for h in range(H):
        cols = slice(h * d_k, (h + 1) * d_k)
        wq = w_qkv[:, :hd][:, cols]
        wk = w_qkv[:, hd:2 * hd][:, cols]
        wv = w_qkv[:, 2 * hd:][:, cols]
        s = np.einsum("bid,bjd->bij", x @ wq, mem @ wk) / math.sqrt(d_k)
        keep = np.ones((B, Lq, Lk), dtype=bool)
        if mask_kind & CAUSAL:
            keep &= np.tril(np.ones((Lq, Lk), dtype=bool))[None]
        if mask_kind & KEYPAD:
            for b in range(B):
                keep[b, :, int(key_lens[b]):] = False
        s = np.where(keep, s, -np.inf)
        m = s.max(axis=-1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.where(keep, np.exp(s - m), 0.0)
        tot = e.sum(axis=-1, keepdims=True)
        a = np.divide(e, tot, out=np.zeros_like(e), where=tot > 0)
        heads.append(a @ (mem @ wv))
    return np.concatenate(heads, axis=-1) @ w_o


def check_torch_mha(layer):
    import torch
    cases = [(1, NONE, False, None), (2, CAUSAL, False, None), (3, KEYPAD, True, [9, 3]),
             (4, BOTH, False, [12, 5]), (5, NONE, True, None)]
    for seed, mask, cross, lens in cases:
        B, H, d_k = 2, 4, 8
        d_model = H * d_k
        Lq = 12
        Lk = 9 if cross else Lq
        x, mem, w_qkv, w_o = _case(seed, B, Lq, Lk, d_model, H, d_k, cross)
        lens_np = np.array(lens, dtype=np.int32) if lens is not None else None
        y = layer(x, w_qkv, w_o, H, mem=mem, mask_kind=mask, key_lens=lens_np)
        mha = torch.nn.MultiheadAttention(d_model, H, bias=False, batch_first=True,
                                          dtype=torch.float64)
        with torch.no_grad():
            mha.in_proj_weight.copy_(torch.from_numpy(w_qkv.T.copy()))
            mha.out_proj.weight.copy_(torch.from_numpy(w_o.T.copy()))
        tx = torch.from_numpy(x)
        tm = torch.from_numpy(mem) if cross else tx
        attn_mask = None
        if mask & CAUSAL:
            attn_mask = ~torch.ones(Lq, Lk, dtype=torch.bool).tril()   # True: not allowed
        kpm = None
        if mask & KEYPAD:
            kpm = torch.arange(Lk)[None, :] >= torch.tensor(lens)[:, None]
        with torch.no_grad():
            ref, _ = mha(tx, tm, tm, attn_mask=attn_mask, key_padding_mask=kpm, need_weights=False)
        assert np.allclose(y, ref.numpy(), rtol=0, atol=1e-12), (seed, np.abs(y - ref.numpy()).max())


def check_identity_weights(layer):
    B, L, H, d_k = 2, 10, 3, 4
    d_model = H * d_k
    rng = np.random.default_rng(7)
    x = rng.standard_normal((B, L, d_model))
    eye = np.eye(d_model)
    w_qkv = np.concatenate([eye, eye, eye], axis=1)
    for mask in (NONE, CAUSAL):
        y = layer(x, w_qkv, eye, H, mask_kind=mask)
        heads = x.reshape(B, L, H, d_k)
        ref = oracle.mha(heads, heads, heads, mask).reshape(B, L, d_model)
        assert np.array_equal(y, ref)


def check_per_head_definition(layer):
    for seed, (mask, cross, lens) in enumerate([(NONE, False, None), (CAUSAL, False, None),
                                                (KEYPAD, True, [11, 1, 6]),
                                                (BOTH, False, [7, 13, 2])]):
        B, H, d_k, d_model = 3, 3, 5, 20       # d_model != H d_k on purpose
        Lq = 13
        Lk = 11 if cross else Lq
        x, mem, w_qkv, w_o = _case(40 + seed, B, Lq, Lk, d_model, H, d_k, cross)
        lens_np = np.array(lens, dtype=np.int32) if lens is not None else None
        y = layer(x, w_qkv, w_o, H, mem=mem, mask_kind=mask, key_lens=lens_np)
        ref = per_head_numpy(x, w_qkv, w_o, H, mem=mem, mask_kind=mask, key_lens=lens_np)
        assert np.allclose(y, ref, rtol=0, atol=1e-12), (mask, np.abs(y - ref).max())


CHECKS = [check_torch_mha, check_identity_weights, check_per_head_definition]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_layer_pin(check):
    check(oracle.mha_layer)


# ---------------------------------------------------------------------------
# planted mistakes: copies of the layer with one thing wrong
# ---------------------------------------------------------------------------
def _layer_variant(mistake):
    def layer(x, w_qkv, w_o, H, mem=None, mask_kind=NONE, key_lens=None):
        x = np.asarray(x, dtype=np.float64)
        mem = x if mem is None else np.asarray(mem, dtype=np.float64)
        B, Lq, d_model = x.shape
        hd = w_qkv.shape[1] // 3
        d_k = hd // H
        wq, wk, wv = w_qkv[:, :hd], w_qkv[:, hd:2 * hd], w_qkv[:, 2 * hd:]
        if mistake == "k_v_blocks_swapped":
            wk, wv = wv, wk
        src_q, src_kv = x, mem
        if mistake == "keys_from_queries":
            src_kv = x
        Lk = src_kv.shape[1]
        q = src_q @ wq
        k = src_kv @ wk
        v = src_kv @ wv
        if mistake == "head_split_transposed":
            q = q.reshape(B, Lq, d_k, H).transpose(0, 1, 3, 2)
            k = k.reshape(B, Lk, d_k, H).transpose(0, 1, 3, 2)
            v = v.reshape(B, Lk, d_k, H).transpose(0, 1, 3, 2)
        else:
            q = q.reshape(B, Lq, H, d_k)
            k = k.reshape(B, Lk, H, d_k)
            v = v.reshape(B, Lk, H, d_k)
        scale = 1.0 / d_k if mistake == "scale_over_dk" else None
        o = oracle.mha(q, k, v, mask_kind, key_lens=key_lens, scale=scale).reshape(B, Lq, hd)
        w = w_o.T if mistake == "w_o_transposed" and w_o.shape[0] == w_o.shape[1] else w_o
        if mistake == "w_o_transposed" and w_o.shape[0] != w_o.shape[1]:
            # not square: the mistake is the head order reversed before W^O
            o = o.reshape(B, Lq, H, d_k)[:, :, ::-1].reshape(B, Lq, hd)
        return o @ w
    return layer


MISTAKES = ["k_v_blocks_swapped", "keys_from_queries", "head_split_transposed",
            "scale_over_dk", "w_o_transposed"]


@pytest.mark.parametrize("mistake", MISTAKES)
def test_layer_mistake_is_caught(mistake):
    layer = _layer_variant(mistake)
    failed = []
    for check in CHECKS:
        try:
            check(layer)
        except (AssertionError, ValueError):
            failed.append(check.__name__)
    assert failed, f"planted mistake {mistake} passed every layer pin"


def test_correct_copy_passes():
    """The copy used for planted mistakes is itself correct without one."""
    layer = _layer_variant("none")
    for check in CHECKS:
        check(layer)
