"""Decode step (mha_decode) vs the float64 oracle through the C ABI.

A decode step is the forward with one query row per sequence and key
lengths = cache lengths, so the oracle is evaluated on q as [B, 1, H, d]
under key padding.  Covers the single-pass and the split (two-kernel) paths,
cache lengths of 0, 1, exact multiples of the 64-key tile and ragged ones,
splits that hold no key, head widths from 8 to 256 (each on the kernel of
the next width up: 64, 128 or 256), the row log-sum-exp, and the decode
workloads at full size on sampled heads.
"""
import zlib

import numpy as np
import pytest
import torch

from tests import parity_util as pu
from transformer_head_scaled_sdpa_gb300 import inputs

pytestmark = pytest.mark.gpu

KEYPAD = inputs.MASK_KEY_PADDING


@pytest.fixture(scope="module")
def mha():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu tests")
    from transformer_head_scaled_sdpa_gb300 import binding, build
    build.build()
    return binding


def make_case(seed, B, H, Lk, d, lens, input_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    case = {}
    for name, shape in (("q", (B, H, d)), ("k_cache", (B, Lk, H, d)), ("v_cache", (B, Lk, H, d))):
        case[name] = (torch.randn(shape, generator=g) * input_scale).to(torch.bfloat16)
    case["cache_lens"] = torch.tensor(lens, dtype=torch.int32)
    return case


def oracle_decode(case, scale=None):
    B, H, d = case["q"].shape
    fwd_case = {"q": case["q"].reshape(B, 1, H, d), "k": case["k_cache"], "v": case["v_cache"],
                "key_lens": case["cache_lens"]}
    out, lse = pu.oracle_run(fwd_case, KEYPAD, scale=scale, return_lse=True)
    return out.reshape(B, H, d), lse.reshape(B, H)


def run(mha, case, scale=0.0):
    g = {n: case[n].cuda() for n in ("q", "k_cache", "v_cache", "cache_lens")}
    out, lse = mha.mha_decode(g["q"], g["k_cache"], g["v_cache"], g["cache_lens"], scale=scale,
                              return_lse=True)
    assert mha.mha_sync_status() == 0
    return out, lse


CASES = [
    # B, H, Lk, d, cache_lens
    (8, 4, 300, 64, [300, 0, 1, 64, 65, 128, 299, 200]),     # split in 2
    (64, 16, 256, 128, None),                                  # one pass
    (1, 2, 5000, 128, [4321]),                                 # 20 splits, the last ones empty
    (4, 8, 1, 64, [1, 0, 1, 1]),
    (3, 2, 8192, 64, [8192, 100, 5000]),                       # 32 splits
    (2, 3, 77, 128, [77, 13]),
    # other head widths: the next kernel width up (64, 128, 256) with the
    # rest of each row read as zero
    (8, 4, 300, 32, [300, 0, 1, 64, 65, 128, 299, 200]),     # split in 2
    (4, 3, 1000, 96, [1000, 999, 64, 3]),                    # split
    (64, 16, 256, 96, None),                                  # one pass
    (2, 4, 3000, 256, [3000, 1234]),                          # split, widest
    (48, 16, 300, 256, None),                                 # one pass, widest
    (3, 5, 130, 8, [130, 129, 0]),                            # narrowest
    (2, 2, 640, 200, [640, 577]),                             # ragged last chunk
]


@pytest.mark.parametrize("shape", CASES, ids=lambda s: "x".join(map(str, s[:4])))
def test_decode_parity(mha, shape):
    B, H, Lk, d, lens = shape
    if lens is None:
        lens = np.random.default_rng(5).integers(1, Lk + 1, size=B).tolist()
    case = make_case(zlib.crc32(repr(shape[:4]).encode()) & 0xFFFF, B, H, Lk, d, lens)
    out, lse = run(mha, case)
    ref, lse_ref = oracle_decode(case)
    pu.assert_bf16_close(out, ref, str(shape[:4]))
    pu.assert_lse_close(lse, lse_ref, str(shape[:4]))
    for b, n in enumerate(lens):
        if n <= 0:
            assert torch.count_nonzero(out[b]) == 0


@pytest.mark.parametrize("scale", [1.0, 0.02])
def test_decode_explicit_scale(mha, scale):
    case = make_case(91, 4, 4, 700, 128, [700, 1, 333, 640])
    out, lse = run(mha, case, scale=scale)
    ref, lse_ref = oracle_decode(case, scale=scale)
    pu.assert_bf16_close_rounding_aware(out, ref, f"scale {scale}")
    pu.assert_lse_close(lse, lse_ref, f"scale {scale}")


def test_decode_matches_padded_rows_ignored(mha):
    """Rows past a cache length do not matter (their weight is exactly 0)."""
    case = make_case(92, 2, 4, 900, 64, [517, 900])
    out1, _ = run(mha, case)
    case["k_cache"][0, 517:] = 7.0
    case["v_cache"][0, 517:] = -3.0
    out2, _ = run(mha, case)
    assert torch.equal(out1, out2)


def test_decode_deterministic_and_workspace_reuse(mha):
    case = make_case(93, 1, 8, 4096, 128, [3000])
    g = {n: case[n].cuda() for n in ("q", "k_cache", "v_cache", "cache_lens")}
    ws = torch.empty(mha.decode_workspace_bytes(1, 8, 4096, 128), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    a = mha.mha_decode(g["q"], g["k_cache"], g["v_cache"], g["cache_lens"], workspace=ws)
    b = mha.mha_decode(g["q"], g["k_cache"], g["v_cache"], g["cache_lens"], workspace=ws)
    assert mha.mha_sync_status() == 0
    assert torch.equal(a, b)
    info = mha.last_launch_info()
    assert info["kernels"] == 2


@pytest.mark.parametrize("name", [w.name for w in inputs.DECODE_WORKLOADS])
def test_decode_workload_sampled_heads(mha, name):
    w = inputs.DECODE_BY_NAME[name]
    case = inputs.generate_decode(w)
    out, lse = run(mha, case)
    out, lse = out.cpu(), lse.cpu()
    rng = np.random.default_rng(w.seed)
    picks = {(0, 0), (w.B - 1, w.H - 1)}
    while len(picks) < 6:
        picks.add((int(rng.integers(w.B)), int(rng.integers(w.H))))
    for b, h in sorted(picks):
        sub = {"q": case["q"][b:b + 1, h:h + 1], "k_cache": case["k_cache"][b:b + 1, :, h:h + 1],
               "v_cache": case["v_cache"][b:b + 1, :, h:h + 1],
               "cache_lens": case["cache_lens"][b:b + 1]}
        sub = {n: t.contiguous() for n, t in sub.items()}
        ref, lse_ref = oracle_decode(sub)
        pu.assert_bf16_close(out[b:b + 1, h:h + 1], ref, f"{name} b={b} h={h}")
        pu.assert_lse_close(lse[b:b + 1, h:h + 1], lse_ref, f"{name} b={b} h={h}")
