"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Covers every workload (in full where the oracle finishes in seconds, else on
sampled heads computed in full by the oracle), ragged and sub-tile shapes,
the three masks, key lengths at 0, 1 and Lk, guard bands around the output,
determinism, causal locality, and the empty cases.
"""
import zlib

import numpy as np
import pytest
import torch

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


# --------------------------------------------------------------------------
# the workloads
# --------------------------------------------------------------------------
SMALL_WORKLOADS = ["toy_cross_f32", "base_encoder_self", "base_decoder_causal",
                   "base_cross_keypad"]
LARGE_WORKLOADS = ["gpt3_causal", "big16_L2048", "big16_L2048_causal", "base8_L4096",
                   "base8_L4096_causal"]


@pytest.mark.parametrize("name", SMALL_WORKLOADS)
def test_workload_full(mha, name):
    w = inputs.BY_NAME[name]
    case = inputs.generate(w)
    out = pu.gpu_run(mha, case, w.mask_kind)
    ref = pu.oracle_run(case, w.mask_kind)
    if w.dtype == torch.float32:
        pu.assert_f32_close(out, ref, name)
        # the toy's heads concatenate to the model width: [1, 4, 2, 3] -> [1, 4, 6]
        assert out.reshape(w.B, w.Lq, w.H * w.d_k).shape == (1, 4, 6)
    else:
        pu.assert_bf16_close(out, ref, name)


@pytest.mark.parametrize("name", LARGE_WORKLOADS)
def test_workload_sampled_heads(mha, name):
    """Full-size launch; the oracle recomputes whole (b, h) heads, sampled."""
    w = inputs.BY_NAME[name]
    case = inputs.generate(w)
    out = pu.gpu_run(mha, case, w.mask_kind).cpu()
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(w.seed)
    picks = {(0, 0), (w.B - 1, w.H - 1)}
    while len(picks) < 4:
        picks.add((int(rng.integers(w.B)), int(rng.integers(w.H))))
    for b, h in sorted(picks):
        sub = {n: case[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v")}
        sub["key_lens"] = case["key_lens"][b:b + 1] if case["key_lens"] is not None else None
        ref = pu.oracle_run(sub, w.mask_kind)
        pu.assert_bf16_close(out[b:b + 1, :, h:h + 1], ref, f"{name} b={b} h={h}")


# --------------------------------------------------------------------------
# shapes: ragged tails, sub-tile, several tiles, both head sizes
# --------------------------------------------------------------------------
SHAPES = [
    # B, H, Lq, Lk, d, mask, key_lens
    (2, 3, 200, 333, 64, NONE, None),
    (2, 3, 200, 333, 128, NONE, None),
    (1, 2, 5, 7, 64, NONE, None),
    (1, 2, 5, 7, 128, NONE, None),
    (2, 2, 256, 1, 64, NONE, None),
    (3, 2, 300, 300, 64, CAUSAL, None),
    (3, 2, 300, 300, 128, CAUSAL, None),
    (2, 4, 129, 129, 64, CAUSAL, None),
    (1, 1, 1, 1, 64, CAUSAL, None),
    (4, 2, 100, 400, 64, KEYPAD, [1, 400, 0, 129]),
    (4, 2, 130, 257, 128, KEYPAD, [257, 128, 127, 1]),
    (2, 3, 384, 640, 64, KEYPAD, [640, 300]),
    (1, 8, 640, 640, 128, NONE, None),
    # d 64 with four or more key tiles and no causal mask: the kernel whose two
    # query tiles take turns at the exponentials (ragged Lq leaves the last
    # unit's second tile empty; ragged Lk masks the last key tile)
    (2, 3, 300, 700, 64, NONE, None),
    (3, 2, 256, 1024, 64, KEYPAD, [1024, 513, 0]),
    # d 64 with at most 128 query rows and more heads than SMs: a unit pairs
    # two heads, each query tile with its own key tiles (odd head counts leave
    # the last unit's second tile empty; key lengths differ between the
    # paired heads)
    (1, 157, 100, 700, 64, NONE, None),
    (3, 53, 128, 1024, 64, KEYPAD, [1024, 0, 385]),
    (5, 33, 128, 300, 64, KEYPAD, [300, 1, 129, 256, 0]),
    (3, 55, 128, 128, 64, CAUSAL, None),
    (2, 77, 77, 77, 64, CAUSAL | KEYPAD, [77, 40]),
    (7, 23, 1, 1000, 64, NONE, None),
    (33, 8, 128, 128, 64, NONE, None),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + f"-m{s[5]}")
def test_shapes(mha, shape):
    B, H, Lq, Lk, d, mask, lens = shape
    case = inputs.random_case(zlib.crc32(repr(shape).encode()) & 0xFFFF, B, H, Lq, Lk, d)
    if lens is not None:
        case["key_lens"] = torch.tensor(lens, dtype=torch.int32)
    out = pu.gpu_run(mha, case, mask)
    ref = pu.oracle_run(case, mask)
    pu.assert_bf16_close(out, ref, str(shape))
    if mask == KEYPAD:
        for b, n in enumerate(lens):
            if n <= 0:
                assert torch.count_nonzero(out[b]) == 0


@pytest.mark.parametrize("scale", [1.0, 0.5, 0.02])
def test_explicit_scale(mha, scale):
    """Explicit scales on N(0, 1) inputs: 1 is unscaled (Luong) attention,
    whose scores have standard deviation 8 at d_k = 64 (formula page, 応用)."""
    case = inputs.random_case(77, 2, 2, 256, 256, 64)
    out = pu.gpu_run(mha, case, NONE, scale=scale)
    ref = pu.oracle_run(case, NONE, scale=scale)
    pu.assert_bf16_close_rounding_aware(out, ref, f"scale {scale}")


@pytest.mark.parametrize("d", [64, 128])
def test_peaked_rows(mha, d):
    """Inputs x2 with scale 1: nearly one-hot rows, |O| up to ~8."""
    case = inputs.random_case(78, 2, 2, 256, 384, d, input_scale=2.0)
    out = pu.gpu_run(mha, case, NONE, scale=1.0)
    ref = pu.oracle_run(case, NONE, scale=1.0)
    pu.assert_bf16_close_rounding_aware(out, ref, f"peaked d={d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", [NONE, CAUSAL])
@pytest.mark.parametrize("step", [8.0, 40.0])
def test_rising_rows(mha, d, mask, step):
    """Scores that climb tile after tile.  Feature 0 of key j is step * (j //
    128) and feature 0 of each query is +-3, so with scale 1 the rows with +3
    climb by 24 (step 8) or 120 (step 40) per 128-key tile, i.e. 35 or 173
    in log2 units (2^173 is past float32's range): every later tile lies far
    above everything before it, so the running maximum moves on every tile,
    while the rows with -3 fall and never move it.  Both kinds share every
    warp."""
    L = 640
    case = inputs.random_case(79, 1, 2, L, L, d)
    g = torch.Generator().manual_seed(80)
    sign = torch.where(torch.rand((1, L, 2), generator=g) < 0.5, -3.0, 3.0)
    case["q"][..., 0] = sign.to(torch.bfloat16)
    tile = (torch.arange(L) // 128).to(torch.float32)
    case["k"][..., 0] = (step * tile).view(1, L, 1).expand(1, L, 2).to(torch.bfloat16)
    out = pu.gpu_run(mha, case, mask, scale=1.0)
    ref = pu.oracle_run(case, mask, scale=1.0)
    assert torch.isfinite(out.float()).all()
    pu.assert_bf16_close_rounding_aware(out, ref, f"rising d={d} mask={mask} step={step}")


# --------------------------------------------------------------------------
# row log-sum-exp (mha_fwd_lse, mha_fwd_f32_lse)
# --------------------------------------------------------------------------
LSE_SHAPES = [
    # B, H, Lq, Lk, d, mask, key_lens, dtype
    (2, 3, 200, 333, 64, NONE, None, torch.bfloat16),
    (2, 3, 300, 700, 64, NONE, None, torch.bfloat16),
    (1, 8, 640, 640, 128, NONE, None, torch.bfloat16),
    (3, 2, 300, 300, 128, CAUSAL, None, torch.bfloat16),
    (2, 4, 129, 129, 64, CAUSAL, None, torch.bfloat16),
    (4, 2, 130, 257, 128, KEYPAD, [257, 0, 127, 1], torch.bfloat16),
    (2, 2, 70, 70, 17, CAUSAL, None, torch.float32),
    (3, 2, 33, 90, 64, KEYPAD, [90, 1, 0], torch.float32),
]


@pytest.mark.parametrize("shape", LSE_SHAPES,
                         ids=lambda s: "x".join(map(str, s[:5])) + f"-m{s[5]}-{str(s[7])[6:]}")
def test_lse(mha, shape):
    """The row log-sum-exp next to the output: -inf exactly on keyless rows,
    else within the float32 bound; the output equals mha_fwd's bit for bit."""
    B, H, Lq, Lk, d, mask, lens, dtype = shape
    case = inputs.random_case(zlib.crc32(repr(shape[:7]).encode()) & 0xFFFF, B, H, Lq, Lk, d,
                              dtype=dtype)
    if lens is not None:
        case["key_lens"] = torch.tensor(lens, dtype=torch.int32)
    out, lse = pu.gpu_run_lse(mha, case, mask)
    ref, lse_ref = pu.oracle_run(case, mask, return_lse=True)
    if dtype == torch.float32:
        pu.assert_f32_close(out, ref, str(shape))
    else:
        pu.assert_bf16_close(out, ref, str(shape))
    pu.assert_lse_close(lse, lse_ref, str(shape))
    assert torch.equal(out, pu.gpu_run(mha, case, mask))


def test_lse_workload_sampled_heads(mha):
    """GPT-3-like workload at full size: lse of sampled whole heads."""
    w = inputs.BY_NAME["gpt3_causal"]
    case = inputs.generate(w)
    _, lse = pu.gpu_run_lse(mha, case, w.mask_kind)
    lse = lse.cpu()
    for b, h in ((0, 0), (w.B - 1, w.H - 1), (1, 37)):
        sub = {n: case[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v")}
        sub["key_lens"] = None
        _, lse_ref = pu.oracle_run(sub, w.mask_kind, return_lse=True)
        pu.assert_lse_close(lse[b:b + 1, h:h + 1], lse_ref, f"gpt3 b={b} h={h}")


@pytest.mark.parametrize("d", [64, 128])
def test_lse_peaked_rows(mha, d):
    """Scale 1 on inputs x2: scores of tens of units, the float32 worst case."""
    case = inputs.random_case(78, 2, 2, 256, 384, d, input_scale=2.0)
    _, lse = pu.gpu_run_lse(mha, case, NONE, scale=1.0)
    _, lse_ref = pu.oracle_run(case, NONE, scale=1.0, return_lse=True)
    pu.assert_lse_close(lse, lse_ref, f"peaked d={d}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_lse_no_keys(mha, dtype):
    """Lk == 0: zero output and lse -inf everywhere."""
    q = torch.randn(2, 5, 3, 64, device="cuda").to(dtype)
    k = torch.empty(2, 0, 3, 64, device="cuda", dtype=dtype)
    fn = mha.mha_fwd if dtype == torch.bfloat16 else mha.mha_fwd_f32
    out = torch.full_like(q, 7.0)
    lse = torch.zeros(2, 3, 5, device="cuda")
    fn(q, k, k, out=out, return_lse=True, lse=lse)
    assert mha.mha_sync_status() == 0
    assert torch.count_nonzero(out) == 0
    assert torch.isneginf(lse).all()


# --------------------------------------------------------------------------
# properties
# --------------------------------------------------------------------------
def test_guard_bands_untouched(mha):
    B, H, Lq, Lk, d = 2, 3, 200, 333, 64
    case = pu.to_cuda(inputs.random_case(5, B, H, Lq, Lk, d))
    n = B * Lq * H * d
    guard = 4096
    buf = torch.full((n + 2 * guard,), 7.25, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n].view(B, Lq, H, d)
    for mask, lens in ((NONE, None), (KEYPAD, torch.tensor([5, 333], dtype=torch.int32).cuda())):
        mha.mha_fwd(case["q"], case["k"], case["v"], out=out, mask_kind=mask, key_lens=lens)
        assert mha.mha_sync_status() == 0
        assert torch.all(buf[:guard] == 7.25) and torch.all(buf[guard + n:] == 7.25)


def test_deterministic(mha):
    case = pu.to_cuda(inputs.random_case(6, 2, 4, 384, 384, 128))
    a = mha.mha_fwd(case["q"], case["k"], case["v"], mask_kind=CAUSAL)
    b = mha.mha_fwd(case["q"], case["k"], case["v"], mask_kind=CAUSAL)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_causal_locality(mha):
    """Output rows <= t do not change when keys/values after t change."""
    case = pu.to_cuda(inputs.random_case(8, 2, 2, 300, 300, 64))
    o = mha.mha_fwd(case["q"], case["k"], case["v"], mask_kind=CAUSAL)
    for t in (0, 127, 128, 200):
        k2 = case["k"].clone()
        v2 = case["v"].clone()
        k2[:, t + 1:] = -3.0
        v2[:, t + 1:] = 5.0
        o2 = mha.mha_fwd(case["q"], k2, v2, mask_kind=CAUSAL)
        torch.cuda.synchronize()
        assert torch.equal(o2[:, :t + 1], o[:, :t + 1]), t


def test_key_padding_ignores_padded_rows(mha):
    case = pu.to_cuda(inputs.random_case(9, 3, 2, 128, 300, 64))
    lens = torch.tensor([300, 77, 129], dtype=torch.int32, device="cuda")
    o = mha.mha_fwd(case["q"], case["k"], case["v"], mask_kind=KEYPAD, key_lens=lens)
    k2 = case["k"].clone()
    v2 = case["v"].clone()
    for b, n in enumerate(lens.tolist()):
        k2[b, n:] = 9.0
        v2[b, n:] = -4.0
    o2 = mha.mha_fwd(case["q"], k2, v2, mask_kind=KEYPAD, key_lens=lens)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)


def test_empty_and_keyless(mha):
    q = torch.zeros((0, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    out = mha.mha_fwd(q, q, q)
    assert out.shape == q.shape
    q = torch.randn((2, 16, 2, 64), device="cuda").to(torch.bfloat16)
    kv = torch.zeros((2, 0, 2, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 3.0)
    mha.mha_fwd(q, kv, kv, out=out)
    assert mha.mha_sync_status() == 0
    assert torch.count_nonzero(out) == 0


@pytest.mark.parametrize("Lq,Lk,d,mask", [(300, 300, 64, NONE), (600, 300, 64, NONE),
                                          (300, 600, 64, NONE), (300, 300, 128, NONE),
                                          (512, 512, 40, NONE), (300, 300, 64, CAUSAL)])
def test_launch_shape(mha, Lq, Lk, d, mask):
    """Heads up to 64 wide over sequences of at most 512 without the causal
    mask take the light one-tile kernel (one 256-thread CTA per (b, h,
    128-query tile)); the rest the two-tile kernel (one 384-thread CTA per
    (b, h, 256 query rows))."""
    case = pu.to_cuda(inputs.random_case(10, 3, 5, Lq, Lk, d))
    mha.mha_fwd(case["q"], case["k"], case["v"], mask_kind=mask)
    info = mha.last_launch_info()
    assert mha.mha_sync_status() == 0
    light = d <= 64 and Lq <= 512 and Lk <= 512 and mask == NONE
    expect = (3 * 5 * ((Lq + 127) // 128), 256) if light else (3 * 5 * ((Lq + 255) // 256), 384)
    assert info["kernels"] == 1 and (info["grid"], info["block"]) == expect, info


@pytest.mark.parametrize("B,H,Lq,d", [(33, 8, 128, 64), (3, 55, 100, 32), (1, 100, 128, 64),
                                      (1, 300, 129, 64), (3, 55, 128, 128)])
def test_paired_launch_shape(mha, B, H, Lq, d):
    """Heads are paired (one CTA per two heads and 128-row query tile) only on
    the two-tile kernel (keys past 512 at widths up to 64), with at most 128
    query rows and more heads than SMs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    case = pu.to_cuda(inputs.random_case(11, B, H, Lq, 600, d))
    mha.mha_fwd(case["q"], case["k"], case["v"])
    info = mha.last_launch_info()
    assert mha.mha_sync_status() == 0
    paired = d <= 64 and Lq <= 128 and B * H > sms
    expect = (B * H + 1) // 2 if paired else B * H * ((Lq + 255) // 256)
    assert info["grid"] == expect, (info, paired, sms)


# --------------------------------------------------------------------------
# float32 path
# --------------------------------------------------------------------------
F32_SHAPES = [
    (1, 2, 4, 8, 3, NONE, None),
    (2, 3, 17, 50, 1, NONE, None),
    (2, 2, 70, 70, 17, CAUSAL, None),
    (3, 2, 33, 90, 64, KEYPAD, [90, 1, 0]),
    (1, 2, 40, 40, 100, CAUSAL, None),
    (2, 1, 20, 65, 256, NONE, None),
]


@pytest.mark.parametrize("shape", F32_SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + f"-m{s[5]}")
def test_f32_shapes(mha, shape):
    B, H, Lq, Lk, d, mask, lens = shape
    case = inputs.random_case(d * 31 + Lk, B, H, Lq, Lk, d, dtype=torch.float32)
    if lens is not None:
        case["key_lens"] = torch.tensor(lens, dtype=torch.int32)
    out = pu.gpu_run(mha, case, mask)
    ref = pu.oracle_run(case, mask)
    pu.assert_f32_close(out, ref, str(shape))


# --------------------------------------------------------------------------
# other head sizes, a value width of its own (d_v != d_k), both masks together
# --------------------------------------------------------------------------
BOTH = inputs.MASK_CAUSAL_KEY_PADDING
WIDTH_SHAPES = [
    # B, H, Lq, Lk, d_k, d_v, mask, key_lens
    (2, 3, 200, 333, 32, 32, NONE, None),
    (2, 2, 300, 700, 32, 32, NONE, None),        # d 64 kernel with exponential turns
    (3, 2, 300, 300, 96, 96, CAUSAL, None),
    (2, 3, 130, 257, 8, 8, KEYPAD, [257, 3]),
    (2, 2, 256, 256, 120, 120, NONE, None),
    (2, 2, 200, 333, 64, 128, NONE, None),
    (2, 2, 256, 256, 128, 64, CAUSAL, None),
    (2, 3, 128, 640, 32, 96, KEYPAD, [640, 100]),
    (1, 4, 100, 100, 48, 16, NONE, None),
    (3, 2, 300, 300, 64, 64, BOTH, [300, 129, 0]),
    (2, 3, 384, 384, 128, 128, BOTH, [200, 384]),
    (2, 2, 1, 1, 64, 64, BOTH, [1, 0]),
    (4, 2, 700, 700, 64, 64, BOTH, [700, 1, 513, 256]),
    (2, 2, 260, 260, 40, 72, BOTH, [260, 77]),
]


def _width_case(shape, dtype=torch.bfloat16):
    B, H, Lq, Lk, d_k, d_v, mask, lens = shape
    case = inputs.random_case(zlib.crc32(repr(shape).encode()) & 0xFFFF, B, H, Lq, Lk, d_k,
                              dtype=dtype, d_v=d_v)
    if lens is not None:
        case["key_lens"] = torch.tensor(lens, dtype=torch.int32)
    return case, mask


@pytest.mark.parametrize("shape", WIDTH_SHAPES,
                         ids=lambda s: "x".join(map(str, s[:6])) + f"-m{s[6]}")
def test_widths_and_both_masks(mha, shape):
    """bf16 on the tensor-core kernels: head sizes other than 64 / 128 run on
    the next wider kernel (tensor maps zero-fill the missing features and clip
    the output), d_v may differ from d_k, and mask kind 3 applies both masks.
    The row log-sum-exp comes out of the same launch."""
    case, mask = _width_case(shape)
    out, lse = pu.gpu_run_lse(mha, case, mask)
    ref, ref_lse = pu.oracle_run(case, mask, return_lse=True)
    assert tuple(out.shape) == ref.shape
    pu.assert_bf16_close(out.cpu(), ref, f"widths {shape}")
    pu.assert_lse_close(lse.cpu(), ref_lse, f"widths {shape}")
    # the plain entry gives the same output bit for bit
    g = pu.to_cuda(case)
    plain = mha.mha_fwd(g["q"], g["k"], g["v"], mask_kind=mask, key_lens=g["key_lens"])
    assert torch.equal(plain, out)


@pytest.mark.parametrize("shape", [(1, 2, 5, 9, 3, 5, NONE, None),
                                   (2, 3, 70, 70, 17, 40, BOTH, [70, 9]),
                                   (2, 2, 33, 90, 64, 8, KEYPAD, [90, 0]),
                                   (1, 2, 40, 40, 256, 200, CAUSAL, None)],
                         ids=lambda s: "x".join(map(str, s[:6])) + f"-m{s[6]}")
def test_f32_widths_and_both_masks(mha, shape):
    case, mask = _width_case(shape, torch.float32)
    out, lse = pu.gpu_run_lse(mha, case, mask)
    ref, ref_lse = pu.oracle_run(case, mask, return_lse=True)
    pu.assert_f32_close(out.cpu(), ref, f"f32 widths {shape}")
    pu.assert_lse_close(lse.cpu(), ref_lse, f"f32 widths {shape}")


def test_both_masks_equal_their_parts(mha):
    """Under both masks, rows below the sequence's key length equal the causal
    launch's rows and rows at or past it equal the key-padding launch's, bit
    for bit (the kernel visits the same keys in the same order)."""
    shape = (3, 2, 520, 520, 64, 64, BOTH, [520, 200, 333])
    case, _ = _width_case(shape)
    both = pu.gpu_run(mha, case, BOTH).cpu()
    causal = pu.gpu_run(mha, case, CAUSAL).cpu()
    pad = pu.gpu_run(mha, case, KEYPAD).cpu()
    for b, n in enumerate(shape[7]):
        assert torch.equal(both[b, :n], causal[b, :n])
        assert torch.equal(both[b, n:], pad[b, n:])


# --------------------------------------------------------------------------
# host-buffer entry and device-side failure reporting
# --------------------------------------------------------------------------
def test_host_entry_matches_device_entry(mha):
    w = inputs.BY_NAME["base_cross_keypad"]
    case = inputs.generate(w)
    dev = pu.gpu_run(mha, case, w.mask_kind).cpu()
    host = {n: case[n].pin_memory() for n in ("q", "k", "v")}
    out = torch.empty_like(host["q"]).pin_memory()
    ws = torch.empty(mha.host_workspace_bytes(w.B, w.H, w.Lq, w.Lk, w.d_k, 2),
                     dtype=torch.uint8, device="cuda")
    mha.mha_fwd_host(host["q"], host["k"], host["v"], out, ws, mask_kind=w.mask_kind,
                     key_lens=case["key_lens"])
    assert torch.equal(out, dev)


@pytest.mark.parametrize("shape", [
    # B, H, Lq, Lk, d, mask, key_lens, dtype.  Below 16 MiB of inputs one
    # chunk; then 8 MiB or more per chunk, up to four: three uneven chunks of
    # five sequences, four of seven (with key padding), two in float32
    (1, 3, 200, 300, 64, NONE, None, torch.bfloat16),
    (5, 2, 33, 90, 40, KEYPAD, [90, 1, 0, 45, 89], torch.float32),
    (5, 16, 512, 512, 128, CAUSAL, None, torch.bfloat16),
    (7, 16, 300, 600, 128, KEYPAD, [600, 0, 1, 128, 129, 300, 599], torch.bfloat16),
    (6, 8, 512, 700, 64, KEYPAD, [700, 1, 0, 350, 699, 128], torch.float32),
], ids=lambda s: "x".join(map(str, s[:5])) + f"-m{s[5]}-{str(s[7])[6:]}")
def test_host_entry_chunks(mha, shape):
    """The host entry runs the batch in chunks of sequences over two streams:
    every sequence's output equals the device entry's, bit for bit."""
    B, H, Lq, Lk, d, mask, lens, dtype = shape
    case = inputs.random_case(zlib.crc32(repr(shape).encode()) & 0xFFFF, B, H, Lq, Lk, d,
                              dtype=dtype)
    if lens is not None:
        case["key_lens"] = torch.tensor(lens, dtype=torch.int32)
    dev = pu.gpu_run(mha, case, mask).cpu()
    host = {n: case[n].pin_memory() for n in ("q", "k", "v")}
    out = torch.full_like(host["q"], 7.0).pin_memory()
    eb = 2 if dtype == torch.bfloat16 else 4
    ws = torch.empty(mha.host_workspace_bytes(B, H, Lq, Lk, d, eb), dtype=torch.uint8,
                     device="cuda")
    mha.mha_fwd_host(host["q"], host["k"], host["v"], out, ws, mask_kind=mask,
                     key_lens=case["key_lens"])
    assert torch.equal(out, dev)


@pytest.mark.parametrize("L,d,mask", [(256, 64, NONE), (256, 64, CAUSAL), (768, 128, CAUSAL),
                                      (300, 256, CAUSAL)])
def test_attention_kernel_timeout_path(mha, L, d, mask):
    """With one pipeline signal withheld, every CTA's bounded wait runs out
    (about a second), the kernel aborts, drains and frees its tensor memory,
    reports MHA_ERR_TIMEOUT, and the next launch computes correctly.  Covers
    the light one-tile kernel (L 256 unmasked), the two-tile kernel at both
    widths and the wide one-tile kernel."""
    case = inputs.random_case(12, 1, 2, L, L, d)
    g = pu.to_cuda(case)
    mha.mha_debug_withhold_p(True)
    try:
        mha.mha_fwd(g["q"], g["k"], g["v"], mask_kind=mask)
        assert mha.mha_sync_status() == 7
    finally:
        mha.mha_debug_withhold_p(False)
    assert mha.mha_sync_status() == 0
    out = pu.gpu_run(mha, case, mask)
    pu.assert_bf16_close(out, pu.oracle_run(case, mask), "after kernel timeout")


def test_attention_kernel_timeout_path_with_turns(mha):
    """The same with the d_k = 64 kernel that passes exponential turns
    between its two query tiles (no mask): the withheld signal still ends in
    MHA_ERR_TIMEOUT, every role leaves, and the next launch is correct."""
    case = inputs.random_case(13, 1, 2, 256, 1024, 64)
    g = pu.to_cuda(case)
    mha.mha_debug_withhold_p(True)
    try:
        mha.mha_fwd(g["q"], g["k"], g["v"], mask_kind=NONE)
        assert mha.mha_sync_status() == 7
    finally:
        mha.mha_debug_withhold_p(False)
    assert mha.mha_sync_status() == 0
    out = pu.gpu_run(mha, case, NONE)
    pu.assert_bf16_close(out, pu.oracle_run(case, NONE), "after kernel timeout")


def test_bounded_wait_reports_timeout(mha):
    """A wait nothing completes gives up (~1 s), reports MHA_ERR_TIMEOUT, and
    the context stays usable."""
    mha.mha_selftest_timeout()
    assert mha.mha_sync_status() == 7
    assert mha.mha_sync_status() == 0  # cleared
    case = inputs.random_case(11, 1, 2, 128, 128, 64)
    out = pu.gpu_run(mha, case, NONE)
    pu.assert_bf16_close(out, pu.oracle_run(case, NONE), "after timeout")
