"""The float64 oracle against what the pages and mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(oracle.mha)


def test_thread_count_changes_no_bit():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((3, 33, 4, 16))
    k = rng.standard_normal((3, 33, 4, 16))
    v = rng.standard_normal((3, 33, 4, 16))
    for mask in (0, 1, 2, 3):
        lens = np.array([33, 5, 0], dtype=np.int32)
        o1 = oracle.mha(q, k, v, mask, key_lens=lens, threads=1)
        o8 = oracle.mha(q, k, v, mask, key_lens=lens, threads=8)
        assert np.array_equal(o1, o8)


def test_bad_arguments_rejected():
    q = np.zeros((1, 3, 1, 4))
    k = np.zeros((1, 5, 1, 4))
    with pytest.raises(ValueError):
        oracle.mha(q, k, k, mask_kind=1)          # causal needs Lq == Lk
    with pytest.raises(ValueError):
        oracle.mha(q, k, k, mask_kind=2)          # key padding needs key_lens
    with pytest.raises(ValueError):
        oracle.mha(q, k, k, mask_kind=5)          # unknown mask kind
    with pytest.raises(ValueError):
        oracle.mha(q, k, k, mask_kind=3, key_lens=np.array([5], dtype=np.int32))  # causal part: Lq == Lk
    qq = np.zeros((1, 5, 1, 4))
    with pytest.raises(ValueError):
        oracle.mha(qq, k, k, mask_kind=3)         # padding part needs key_lens


def test_value_width_below_key_width():
    """d_v < d_k against the brute force and torch's float64 SDPA (kept out of
    the planted-mistake runs, whose stride mutants would read past v here)."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(16)
    for mask in (0, 3):
        B, L, H, d_k, d_v = 2, 5, 2, 6, 2
        q = rng.standard_normal((B, L, H, d_k))
        k = rng.standard_normal((B, L, H, d_k))
        v = rng.standard_normal((B, L, H, d_v))
        lens = np.array([5, 2], dtype=np.int32) if mask & 2 else None
        o = oracle.mha(q, k, v, mask, key_lens=lens)
        assert o.shape == (B, L, H, d_v)
        assert np.allclose(o, oracle_pins.brute_force(q, k, v, mask, lens), rtol=0, atol=1e-12)
        allowed = torch.ones(B, 1, L, L, dtype=torch.bool)
        if mask & 1:
            allowed &= torch.ones(L, L, dtype=torch.bool).tril()
        if mask & 2:
            for b in range(B):
                allowed[b, :, :, int(lens[b]):] = False
        tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=allowed).permute(0, 2, 1, 3)
        assert np.allclose(o, ref.numpy(), rtol=0, atol=1e-12)
