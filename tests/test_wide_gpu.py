"""Heads wider than 128 features (d_k, d_v up to 256: the wide kernel), the
light 64-wide variant of the same one-tile kernel (short unmasked or
key-padded sequences), and heads narrower than the 64- and 128-wide kernels
(which issue only their own K steps and output columns), against the float64
oracle through the C ABI.

Covers every mask kind, ragged query and key lengths (several 64-key tiles,
a ragged last one, sub-tile shapes), key lengths 0 and 1, d_v != d_k in both
directions, the row log-sum-exp, scores that climb tile after tile (the
running maximum moves every tile, so O is rescaled), causal locality and
padded-key invariance (bit-exact), more units than SMs, and a full-size
d_k = 256 causal launch checked on sampled heads.
"""
import zlib

import numpy as np
import pytest
import torch

from tests import parity_util as pu
from transformer_head_scaled_sdpa_gb300 import inputs

pytestmark = pytest.mark.gpu

NONE, CAUSAL, KEYPAD, BOTH = 0, 1, 2, 3


@pytest.fixture(scope="module")
def mha():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu tests")
    from transformer_head_scaled_sdpa_gb300 import binding, build
    build.build()
    return binding


def _case(shape):
    B, H, Lq, Lk, d_k, d_v, mask, lens = shape
    case = inputs.random_case(zlib.crc32(repr(shape).encode()) & 0xFFFF, B, H, Lq, Lk, d_k,
                              d_v=d_v)
    if lens is not None:
        case["key_lens"] = torch.tensor(lens, dtype=torch.int32)
    return case


SHAPES = [
    # B, H, Lq, Lk, d_k, d_v, mask, key_lens
    (2, 3, 200, 333, 256, 256, NONE, None),
    (1, 2, 5, 7, 256, 256, NONE, None),
    (3, 2, 300, 300, 256, 256, CAUSAL, None),
    (2, 2, 129, 129, 256, 256, CAUSAL, None),
    (4, 2, 130, 257, 256, 256, KEYPAD, [257, 64, 0, 1]),
    (2, 3, 150, 150, 256, 256, BOTH, [150, 63]),
    (2, 2, 256, 700, 192, 192, NONE, None),
    (2, 2, 190, 190, 136, 136, CAUSAL, None),
    (2, 2, 100, 300, 256, 64, NONE, None),        # d_v < d_k
    (2, 2, 100, 300, 64, 256, KEYPAD, [300, 33]),  # d_v > d_k
    (1, 3, 70, 90, 160, 248, NONE, None),
    (1, 200, 64, 200, 256, 256, NONE, None),       # more units than SMs
    # narrow heads on the 64- and 128-wide kernels (their own K steps and
    # output columns)
    (2, 3, 200, 333, 32, 32, NONE, None),
    (2, 3, 300, 300, 96, 96, CAUSAL, None),
    (2, 2, 130, 700, 40, 40, KEYPAD, [700, 129]),
    (1, 160, 100, 300, 32, 32, NONE, None),        # paired heads, narrow
    (2, 2, 300, 700, 32, 32, NONE, None),
    (2, 2, 200, 200, 128, 48, CAUSAL, None),
    (2, 2, 200, 200, 80, 112, NONE, None),
    # the light one-tile kernel (heads up to 64 wide, sequences up to 512, no
    # causal mask): d_v != d_k, key padding, ragged tiles, a one-wave grid
    # (early trigger of the next launch) and more units than CTA slots
    (2, 3, 300, 400, 64, 32, NONE, None),
    (2, 2, 256, 512, 48, 64, KEYPAD, [512, 77]),
    (1, 2, 1, 1, 64, 64, NONE, None),
    (2, 8, 128, 128, 64, 64, NONE, None),
    (1, 400, 128, 130, 64, 64, KEYPAD, [129]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:6])) + f"-m{s[6]}")
def test_widths(mha, shape):
    case = _case(shape)
    mask, lens = shape[6], shape[7]
    out, lse = pu.gpu_run_lse(mha, case, mask)
    ref, lse_ref = pu.oracle_run(case, mask, return_lse=True)
    pu.assert_bf16_close(out, ref, str(shape))
    pu.assert_lse_close(lse, lse_ref, str(shape))
    if lens is not None:
        for b, n in enumerate(lens):
            if n <= 0:
                assert torch.count_nonzero(out[b]) == 0


@pytest.mark.parametrize("mask", [NONE, CAUSAL])
def test_wide_rising_rows(mha, mask):
    """Feature 0 of key j is 8 * (j // 64) and feature 0 of each query +-3, so
    with scale 1 the +3 rows climb by 35 log2 units per 64-key tile: the
    running maximum moves on every tile and O is rescaled each time."""
    L, d = 512, 256
    case = inputs.random_case(81, 1, 2, L, L, d)
    g = torch.Generator().manual_seed(82)
    sign = torch.where(torch.rand((1, L, 2), generator=g) < 0.5, -3.0, 3.0)
    case["q"][..., 0] = sign.to(torch.bfloat16)
    tile = (torch.arange(L) // 64).to(torch.float32)
    case["k"][..., 0] = (8.0 * tile).view(1, L, 1).expand(1, L, 2).to(torch.bfloat16)
    out = pu.gpu_run(mha, case, mask, scale=1.0)
    ref = pu.oracle_run(case, mask, scale=1.0)
    assert torch.isfinite(out.float()).all()
    pu.assert_bf16_close_rounding_aware(out, ref, f"wide rising mask={mask}")


def test_light_launch_back_to_back(mha):
    """Consecutive launches of the light kernel on one stream (the one-wave
    grid triggers the next launch at its start; each launch still waits for
    the previous one before it touches global memory): every output matches
    the oracle, including a launch that overwrites the previous one's output
    buffer and one that reads it as its input."""
    host = inputs.random_case(86, 2, 8, 128, 128, 64)
    case = pu.to_cuda(host)
    ref = pu.oracle_run(host, NONE)
    outs = [mha.mha_fwd(case["q"], case["k"], case["v"]) for _ in range(4)]
    same = torch.empty_like(case["q"])
    for _ in range(3):
        mha.mha_fwd(case["q"], case["k"], case["v"], out=same)
    # the next launch reads the previous launch's output as its values
    chained = mha.mha_fwd(case["q"], case["k"], same)
    assert mha.mha_sync_status() == 0
    for o in outs + [same]:
        pu.assert_bf16_close(o.cpu(), ref, "light back to back")
    host2 = {"q": host["q"], "k": host["k"], "v": same.cpu(), "key_lens": None}
    pu.assert_bf16_close(chained.cpu(), pu.oracle_run(host2, NONE), "light chained")


def test_wide_causal_locality(mha):
    case = pu.to_cuda(inputs.random_case(83, 2, 2, 300, 300, 256))
    o = mha.mha_fwd(case["q"], case["k"], case["v"], mask_kind=CAUSAL)
    for t in (0, 63, 64, 127, 128, 250):
        k2 = case["k"].clone()
        v2 = case["v"].clone()
        k2[:, t + 1:] = -3.0
        v2[:, t + 1:] = 5.0
        o2 = mha.mha_fwd(case["q"], k2, v2, mask_kind=CAUSAL)
        torch.cuda.synchronize()
        assert torch.equal(o2[:, :t + 1], o[:, :t + 1]), t


def test_wide_padding_ignored_and_deterministic(mha):
    case = pu.to_cuda(inputs.random_case(84, 3, 2, 128, 300, 256))
    lens = torch.tensor([300, 77, 129], dtype=torch.int32, device="cuda")
    o = mha.mha_fwd(case["q"], case["k"], case["v"], mask_kind=KEYPAD, key_lens=lens)
    o_again = mha.mha_fwd(case["q"], case["k"], case["v"], mask_kind=KEYPAD, key_lens=lens)
    k2 = case["k"].clone()
    v2 = case["v"].clone()
    for b, n in enumerate(lens.tolist()):
        k2[b, n:] = 9.0
        v2[b, n:] = -4.0
    o2 = mha.mha_fwd(case["q"], k2, v2, mask_kind=KEYPAD, key_lens=lens)
    assert mha.mha_sync_status() == 0
    assert torch.equal(o, o_again)
    assert torch.equal(o, o2)


def test_wide_full_size_sampled_heads(mha):
    """A d_k = 256 causal launch of 2 x 16 heads at L 2048 (512 units, over
    three per SM), checked on sampled whole heads."""
    B, H, L, d = 2, 16, 2048, 256
    case = inputs.random_case(85, B, H, L, L, d)
    out = pu.gpu_run(mha, case, CAUSAL).cpu()
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(85)
    picks = {(0, 0), (B - 1, H - 1)}
    while len(picks) < 4:
        picks.add((int(rng.integers(B)), int(rng.integers(H))))
    for b, h in sorted(picks):
        sub = {n: case[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v")}
        sub["key_lens"] = None
        ref = pu.oracle_run(sub, CAUSAL)
        pu.assert_bf16_close(out[b:b + 1, :, h:h + 1], ref, f"d256 b={b} h={h}")


def test_wide_random_sweep(mha):
    """Seeded random sizes, masks and widths from 136 to 256."""
    r = np.random.default_rng(4242)
    for i in range(12):
        mask = int(r.integers(0, 4))
        B, H = int(r.integers(1, 3)), int(r.integers(1, 4))
        Lq = int(r.integers(1, 400))
        Lk = Lq if mask & CAUSAL else int(r.integers(1, 400))
        d_k = int(r.choice([136, 144, 200, 256]))
        d_v = d_k if r.random() < 0.5 else int(r.choice([8, 64, 136, 256]))
        lens = r.integers(0, Lk + 1, size=B).tolist() if mask & KEYPAD else None
        shape = (B, H, Lq, Lk, d_k, d_v, mask, lens)
        case = _case(shape)
        out = pu.gpu_run(mha, case, mask)
        ref = pu.oracle_run(case, mask)
        pu.assert_bf16_close_rounding_aware(out, ref, str(shape))
