"""mha_decode_static: the decode step with the library's fixed device scratch
instead of a caller workspace.

On the GPU it must give exactly what mha_decode gives, call after call (two
consecutive calls of each, on a split and a one-pass case).  On the host,
every size the decode accepts (head widths up to 256) must fit the fixed
array.
"""
import pytest
import torch

from transformer_head_scaled_sdpa_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def test_static_scratch_covers_every_decode_size(lib):
    """The split count keeps the partials small: check the workspace need
    against the fixed array for every head count that splits and cache
    lengths up to far past any context."""
    cap = lib.mha_decode_static_scratch_bytes()
    assert cap == 2 << 20
    worst = 0
    for bh in range(1, 700):
        for lk in (1, 255, 256, 257, 1000, 4096, 16384, 1 << 20):
            for d in (8, 64, 96, 128, 200, 256):
                worst = max(worst, lib.mha_decode_workspace_bytes(1, bh, lk, d))
    assert 0 < worst <= cap


def make(seed, B, H, Lk, d, lens):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, Lk, H, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, Lk, H, d, generator=g).to(torch.bfloat16).cuda()
    return q, k, v, torch.tensor(lens, dtype=torch.int32).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 8, 4096, 128, [3001]),          # split: 16 chunks
                                   (2, 3, 700, 64, [700, 129]),        # split: 3 chunks
                                   (64, 16, 256, 128, [200] * 64),     # one pass
                                   (3, 5, 1500, 256, [1500, 7, 700]),  # split, d_k 256
                                   (4, 2, 900, 40, [900, 1, 5, 333])],  # split, d_k 40
                         ids=["split16", "split3", "onepass", "split_d256", "split_d40"])
def test_static_matches_workspace_entry(lib, shape):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu tests")
    B, H, Lk, d, lens = shape
    q, k, v, lens_d = make(17, B, H, Lk, d, lens)
    got = []
    for _ in range(2):   # two consecutive calls of each entry
        o_ws, l_ws = binding.mha_decode(q, k, v, lens_d, return_lse=True)
        o_st, l_st = binding.mha_decode_static(q, k, v, lens_d, return_lse=True)
        assert binding.mha_sync_status() == 0
        got.append((o_ws, l_ws, o_st, l_st))
    for o_ws, l_ws, o_st, l_st in got:
        assert torch.equal(o_st, o_ws)
        assert torch.equal(l_st, l_ws)
    assert torch.equal(got[0][2], got[1][2]) and torch.equal(got[0][3], got[1][3])
    assert torch.isfinite(got[0][3]).all()
