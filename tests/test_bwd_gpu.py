"""Gradient (mha_bwd) vs the float64 oracle's gradient, through the C ABI.

The GPU runs mha_fwd_lse and then mha_bwd on the same bf16 inputs; the oracle
recomputes the forward and the gradient in float64 from those inputs and the
same dout.  Covers one tile, ragged tails in both lengths, both head sizes,
the three masks (key lengths 0, 1, Lk and ragged), keys no query sees
(zero gradient), and sampled heads of the GPT-3-like workload at full size.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from tests import parity_util as pu
from transformer_head_scaled_sdpa_gb300 import inputs

pytestmark = pytest.mark.gpu

NONE, CAUSAL, KEYPAD = inputs.MASK_NONE, inputs.MASK_CAUSAL, inputs.MASK_KEY_PADDING


@pytest.fixture(scope="module")
def mha():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu tests")
    from transformer_head_scaled_sdpa_gb300 import binding, build
    build.build()
    return binding


def run_bwd(mha, case, dout, mask, scale=0.0):
    g = pu.to_cuda(case)
    out, lse = mha.mha_fwd(g["q"], g["k"], g["v"], mask_kind=mask, key_lens=g["key_lens"],
                           scale=scale, return_lse=True)
    dq, dk, dv = mha.mha_bwd(g["q"], g["k"], g["v"], out, dout.cuda(), lse, mask_kind=mask,
                             key_lens=g["key_lens"], scale=scale)
    assert mha.mha_sync_status() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


def grad_errors(got, ref):
    """(max |g - ref| / max |ref|, ||g - ref||_F / ||ref||_F)"""
    g = got.to(torch.float64).numpy()
    scale = float(np.abs(ref).max()) or 1.0
    fro = float(np.linalg.norm(ref)) or 1.0
    return float(np.abs(g - ref).max()) / scale, float(np.linalg.norm(g - ref)) / fro


SHAPES = [
    # B, H, Lq, Lk, d, mask, key_lens
    (1, 2, 128, 128, 64, NONE, None),
    (2, 3, 200, 333, 64, NONE, None),
    (1, 2, 256, 256, 128, NONE, None),
    (1, 1, 5, 7, 64, NONE, None),
    (3, 2, 300, 300, 128, CAUSAL, None),
    (2, 4, 129, 129, 64, CAUSAL, None),
    (4, 2, 130, 257, 128, KEYPAD, [257, 0, 127, 1]),
    # both masks together (kind 3); other head sizes on the 64 / 128 kernels
    (3, 2, 300, 300, 64, 3, [300, 129, 0]),
    (2, 2, 256, 256, 128, 3, [200, 256]),
    (2, 3, 200, 333, 32, NONE, None),
    (3, 2, 300, 300, 96, CAUSAL, None),
    (2, 2, 130, 257, 8, KEYPAD, [257, 40]),
    # more units than SMs, so every CTA runs several units back to back (the
    # kernels are persistent), with units without keys between them, rows
    # past Lk clipped by the dK/dV tensor-map stores, and dQ rows on both
    # store paths (whole 32-byte sectors at d 128, 16-byte stores at d 40)
    (5, 40, 256, 256, 64, KEYPAD, [256, 0, 130, 1, 255]),
    (3, 60, 300, 300, 128, 3, [300, 0, 129]),
    (2, 80, 200, 333, 128, NONE, None),
    (4, 40, 150, 150, 40, CAUSAL, None),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + f"-m{s[5]}")
def test_bwd_parity(mha, shape):
    B, H, Lq, Lk, d, mask, lens = shape
    seed = zlib.crc32(repr(shape).encode()) & 0xFFFF
    case = inputs.random_case(seed, B, H, Lq, Lk, d)
    if lens is not None:
        case["key_lens"] = torch.tensor(lens, dtype=torch.int32)
    dout = inputs.random_case(seed + 1, B, H, Lq, Lq, d)["q"]
    got = run_bwd(mha, case, dout, mask)
    ref = oracle.mha_bwd(case["q"], case["k"], case["v"], dout, mask,
                         key_lens=case["key_lens"].numpy() if lens is not None else None)
    for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
        assert torch.isfinite(gg.float()).all(), name
        rel_max, rel_fro = grad_errors(gg, rr)
        print(f"{shape} {name}: max {rel_max:.2e} fro {rel_fro:.2e}")
        assert rel_max <= pu.BWD_REL_MAX and rel_fro <= pu.BWD_REL_FRO, \
            f"{shape} {name}: max {rel_max:.3e} fro {rel_fro:.3e}"
    if mask == KEYPAD:
        for b, n in enumerate(lens):
            assert torch.count_nonzero(got[1][b, max(n, 0):]) == 0
            assert torch.count_nonzero(got[2][b, max(n, 0):]) == 0


def test_bwd_workload_sampled_heads(mha):
    """GPT-3-like workload at full size; two whole heads against the oracle."""
    w = inputs.BY_NAME["gpt3_causal"]
    case = inputs.generate(w)
    dout = inputs.generate(w, seed=w.seed + 77)["q"]
    got = run_bwd(mha, case, dout, w.mask_kind)
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        sub = {n: case[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v")}
        ref = oracle.mha_bwd(sub["q"], sub["k"], sub["v"], dout[b:b + 1, :, h:h + 1].contiguous(),
                             w.mask_kind)
        for name, gg, rr in zip(("dq", "dk", "dv"), got, ref):
            rel_max, rel_fro = grad_errors(gg[b:b + 1, :, h:h + 1], rr)
            print(f"gpt3 b={b} h={h} {name}: max {rel_max:.2e} fro {rel_fro:.2e}")
            assert rel_max <= pu.BWD_REL_MAX and rel_fro <= pu.BWD_REL_FRO, \
                f"gpt3 {name}: max {rel_max:.3e} fro {rel_fro:.3e}"
