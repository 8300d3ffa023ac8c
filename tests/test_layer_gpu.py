"""The multi-head layer (mha_layer_fwd: the library's tensor-core GEMM for
the projections around the attention kernel) against the float64 layer
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
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


def _run(mha, case, H, mask):
    dev = {n: (t.cuda() if t is not None else None) for n, t in case.items()}
    y = mha.mha_layer_fwd(dev["x"], dev["w_qkv"], dev["w_o"], H, mem=dev["mem"], mask_kind=mask,
                          key_lens=dev["key_lens"])
    assert mha.mha_sync_status() == 0
    return y.cpu()


def _oracle(case, H, mask):
    lens = case["key_lens"].numpy() if case["key_lens"] is not None else None
    return oracle.mha_layer(case["x"], case["w_qkv"], case["w_o"], H, mem=case["mem"],
                            mask_kind=mask, key_lens=lens)


@pytest.mark.parametrize("name", ["base_layer_decoder", "base_layer_cross"])
def test_layer_workloads(mha, name):
    w = inputs.LAYER_BY_NAME[name]
    case = inputs.generate_layer(w)
    y = _run(mha, case, w.H, w.mask_kind)
    pu.assert_layer_close(y, _oracle(case, w.H, w.mask_kind), name)


SHAPES = [
    # B, Lq, Lk, d_model, H, d_k, mask, cross, key_lens
    (2, 200, 200, 256, 4, 64, CAUSAL, False, None),
    (2, 130, 300, 256, 2, 128, KEYPAD, True, [300, 7]),
    (3, 150, 150, 192, 6, 32, BOTH, False, [150, 64, 1]),
    (1, 5, 9, 64, 2, 32, NONE, True, None),
    (2, 260, 260, 384, 3, 96, NONE, False, None),      # d_model != H d_k
    (1, 256, 256, 4096, 32, 128, CAUSAL, False, None),  # K 4096: 256-row GEMM tiles
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:6])) + f"-m{s[6]}")
def test_layer_shapes(mha, shape):
    B, Lq, Lk, d_model, H, d_k, mask, cross, lens = shape
    # seeded with the workloads' recipe (x, mem, w_qkv, w_o), without a registered name
    g = torch.Generator().manual_seed(4000 + sum(shape[:6]))
    x = torch.randn((B, Lq, d_model), generator=g)
    mem = torch.randn((B, Lk, d_model), generator=g) if cross else None
    w_qkv = torch.randn((d_model, 3 * H * d_k), generator=g) * d_model ** -0.5
    w_o = torch.randn((H * d_k, d_model), generator=g) * (H * d_k) ** -0.5
    case = {"x": x.to(torch.bfloat16), "mem": mem.to(torch.bfloat16) if cross else None,
            "w_qkv": w_qkv.to(torch.bfloat16), "w_o": w_o.to(torch.bfloat16),
            "key_lens": torch.tensor(lens, dtype=torch.int32) if lens is not None else None}
    y = _run(mha, case, H, mask)
    pu.assert_layer_close(y, _oracle(case, H, mask), f"layer {shape}")


def test_layer_gpt3_sampled_rows(mha):
    """The GPT-3-like layer at full size (one sequence): under the causal mask
    rows 0 .. 255 depend only on x rows 0 .. 255, so the oracle computes them on
    that prefix exactly."""
    w = inputs.LAYER_BY_NAME["gpt3_layer_b1"]
    case = inputs.generate_layer(w)
    y = _run(mha, case, w.H, w.mask_kind)
    n = 256
    sub = dict(case, x=case["x"][:, :n].contiguous())
    ref = _oracle(sub, w.H, w.mask_kind)
    pu.assert_layer_close(y[:, :n], ref, "gpt3 layer, rows 0..255")
    assert torch.isfinite(y.to(torch.float32)).all()


def test_layer_self_equals_cross_with_itself(mha):
    """Self-attention (mem NULL: one packed Q|K|V GEMM) and cross-attention
    with the memory set to x (two GEMMs over the weight's column blocks) give
    the same layer output."""
    w = inputs.LAYER_BY_NAME["base_layer_decoder"]
    case = inputs.generate_layer(w)
    y_self = _run(mha, case, w.H, w.mask_kind)
    y_cross = _run(mha, dict(case, mem=case["x"].clone()), w.H, w.mask_kind)
    ref = _oracle(case, w.H, w.mask_kind)
    pu.assert_layer_close(y_cross, ref, "cross with itself")
    # both round the same projections; GEMM split orders may differ slightly
    assert float((y_self.float() - y_cross.float()).abs().max()) <= 2 ** -6 * float(np.abs(ref).max())
