"""The tensor-core GEMM of the layer's projections (mha_gemm_bf16) against a
float32 product of the same bf16 operands, through the C ABI.

The kernel accumulates in float32 and rounds each result once to bf16, so
against a float32 (or float64) product of the same inputs the error is the
output rounding (half a bf16 unit, 2^-9 relative) plus float32 summation
differences: each element within 2^-8 of its magnitude plus 2^-14 of the
largest, and the whole within 2^-9 relative Frobenius.  Shapes cover single
tiles, ragged edges in M, N and K, strided row views (the layer reads column
blocks of the packed weight in place), more tiles than SMs, K = 0, and both
tilings (128-row tiles below K = 4096, 256-row tiles from there on).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mha():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu tests")
    from transformer_head_scaled_sdpa_gb300 import binding, build
    build.build()
    return binding


def _operands(seed, M, N, K, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn(M, K, generator=g) * scale).to(torch.bfloat16)
    b = (torch.randn(K, N, generator=g) / max(K, 1) ** 0.5).to(torch.bfloat16)
    return a, b


def _check(got, ref, what):
    got = got.double().cpu()
    ref = ref.double().cpu()
    err = (got - ref).abs()
    bound = 2.0 ** -8 * ref.abs() + 2.0 ** -14 * ref.abs().max()
    worst = float((err - bound).max())
    assert worst <= 0, f"{what}: element error exceeds the bound by {worst:.3e}"
    rel = float(torch.linalg.norm(got - ref) / max(float(torch.linalg.norm(ref)), 1e-30))
    assert rel <= 2.0 ** -9, f"{what}: relative Frobenius {rel:.3e}"


SHAPES = [
    (1, 8, 8), (128, 256, 64), (100, 200, 72), (300, 520, 200), (257, 1000, 1032),
    (1024, 768, 512), (2048, 1536, 512), (96, 4104, 40),
    # K >= 4096: 256-row tiles (two accumulators), ragged in M, N and K
    (300, 520, 4104), (129, 264, 4096), (513, 776, 6152),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_matches_float64_product(mha, shape):
    """Three calls each (a staging buffer reused before its store has read it
    would show as a call that differs)."""
    M, N, K = shape
    a, b = _operands(sum(shape), M, N, K)
    a, b = a.cuda(), b.cuda()
    ref = a.double().cpu() @ b.double().cpu()
    outs = [mha.mha_gemm_bf16(a, b) for _ in range(3)]
    assert mha.mha_sync_status() == 0
    for i, c in enumerate(outs):
        _check(c, ref, f"{shape} call {i}")


def test_gemm_large_against_float32(mha):
    """Many more tiles than SMs, over a long K (a GPT-3-like projection's K)."""
    M, N, K = 4096, 6144, 12288
    a, b = _operands(7, M, N, K)
    a, b = a.cuda(), b.cuda()
    c = mha.mha_gemm_bf16(a, b)
    ref = a.float() @ b.float()
    assert mha.mha_sync_status() == 0
    _check(c, ref, "4096x6144x12288")


def test_gemm_strided_views(mha):
    """Column blocks of wider row-major matrices, read and written in place."""
    M, N, K = 300, 192, 264
    a, w = _operands(11, M, 3 * N, K)
    w = w.cuda()
    base = torch.zeros(M, 2 * N + 8, dtype=torch.bfloat16, device="cuda")
    c = base[:, 8:8 + N]                        # a view with row stride 2N + 8
    a_wide = torch.zeros(M, K + 40, dtype=torch.bfloat16, device="cuda")
    a_wide[:, :K] = a.cuda()
    b_view = w[:, N:2 * N]                      # the middle column block, row stride 3N
    mha.mha_gemm_bf16(a_wide[:, :K], b_view, c)
    assert mha.mha_sync_status() == 0
    _check(c, a.double() @ w[:, N:2 * N].double().cpu(), "strided")
    assert torch.count_nonzero(base[:, :8]) == 0 and torch.count_nonzero(base[:, 8 + N:]) == 0


def test_gemm_empty_k_writes_zeros(mha):
    a = torch.empty(5, 0, dtype=torch.bfloat16, device="cuda")
    b = torch.empty(0, 16, dtype=torch.bfloat16, device="cuda")
    c = torch.full((5, 16), 3.0, dtype=torch.bfloat16, device="cuda")
    mha.mha_gemm_bf16(a, b, c)
    assert mha.mha_sync_status() == 0
    assert torch.count_nonzero(c) == 0


def test_gemm_deterministic(mha):
    a, b = _operands(3, 700, 904, 1096)
    a, b = a.cuda(), b.cuda()
    c1 = mha.mha_gemm_bf16(a, b)
    c2 = mha.mha_gemm_bf16(a, b)
    assert mha.mha_sync_status() == 0
    assert torch.equal(c1, c2)
