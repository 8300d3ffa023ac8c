"""The C ABI on the host: libmha.so builds, loads, exports every function
include/*.h declares, and rejects bad arguments with the documented codes.
The argument checks run before any CUDA call, so no GPU is needed; pointers
below are never dereferenced."""
import ctypes
import math
import os
import re

import pytest

from transformer_head_scaled_sdpa_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", n) for n in sorted(os.listdir(os.path.join(ROOT, "include")))
           if n.endswith(".h")]

OK, NULL, SHAPE, UNSUP, MASK, SCALE, LAUNCH, TIMEOUT, ALIAS, WORKSPACE = range(10)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    names = set()
    for path in HEADERS:
        text = open(path, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(mha_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mha_fwd" in names and "mha_fwd_f32" in names and "mha_sync_status" in names
    assert "mha_debug_withhold_p" in names and "mha_gemm_bf16" in names
    raw = ctypes.CDLL(binding.library_path())
    for n in names:
        assert hasattr(raw, n), f"libmha.so does not export {n}"


def test_status_strings(lib):
    for code in range(10):
        s = binding.mha_status_string(code)
        assert s and s != "unknown status"
    assert binding.mha_status_string(99) == "unknown status"


# fake, 256-aligned, non-overlapping device addresses
Q, K, V, O, LENS = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def fwd(lib, fn="mha_fwd", q=Q, k=K, v=V, o=O, B=2, H=3, Lq=64, Lk=64, d=64, mask=0,
        lens=None, scale=0.0):
    return getattr(lib, fn)(q, k, v, o, B, H, Lq, Lk, d, mask, lens, scale, None)


@pytest.mark.parametrize("fn", ["mha_fwd", "mha_fwd_f32"])
def test_argument_errors(lib, fn):
    assert fwd(lib, fn, B=-1) == SHAPE
    assert fwd(lib, fn, Lk=-5) == SHAPE
    assert fwd(lib, fn, d=0) == SHAPE
    assert fwd(lib, fn, mask=1, Lq=64, Lk=65) == SHAPE          # causal needs Lq == Lk
    assert fwd(lib, fn, mask=4) == MASK                           # unknown mask kind
    assert fwd(lib, fn, mask=-1) == MASK
    assert fwd(lib, fn, mask=2, lens=None) == MASK               # key padding needs key_lens
    assert fwd(lib, fn, mask=3, lens=None) == MASK               # so do both masks together
    assert fwd(lib, fn, mask=3, lens=LENS, Lq=64, Lk=65) == SHAPE  # and the causal part Lq == Lk
    assert fwd(lib, fn, scale=math.nan) == SCALE
    assert fwd(lib, fn, scale=math.inf) == SCALE
    assert fwd(lib, fn, scale=-0.5) == SCALE
    assert fwd(lib, fn, q=None) == NULL
    assert fwd(lib, fn, o=None) == NULL
    assert fwd(lib, fn, k=None) == NULL
    assert fwd(lib, fn, o=Q + 64) == ALIAS                        # out overlaps q
    assert fwd(lib, fn, o=K) == ALIAS
    assert fwd(lib, fn, B=1 << 20, H=1 << 10, Lq=1 << 20) == SHAPE  # row count overflow
    # empty query side: nothing to do, no device touched
    assert fwd(lib, fn, B=0) == OK
    assert fwd(lib, fn, Lq=0, mask=0) == OK
    assert fwd(lib, fn, H=0, q=None, o=None) == OK


def test_bf16_specific_errors(lib):
    assert fwd(lib, d=12) == UNSUP          # bf16 path: d_k a multiple of 8 ...
    assert fwd(lib, d=4) == UNSUP
    assert fwd(lib, d=264) == UNSUP         # ... up to 256
    assert fwd(lib, d=260) == UNSUP
    assert fwd(lib, q=Q + 8) == UNSUP       # TMA needs 16-byte aligned bases
    assert fwd(lib, fn="mha_fwd_f32", d=257) == UNSUP
    assert fwd(lib, fn="mha_fwd_f32", q=Q + 2) == UNSUP


def test_host_entry_errors(lib):
    assert lib.mha_fwd_host_workspace_bytes(2, 3, 64, 64, 64, 2) > 0
    assert lib.mha_fwd_host_workspace_bytes(2, 3, 64, 64, 64, 3) == 0
    assert lib.mha_fwd_host(Q, K, V, O, 2, 3, 64, 64, 64, 0, None, 0.0, 2, None, 0, None) == WORKSPACE
    assert lib.mha_fwd_host(Q, K, V, O, 2, 3, 64, 64, 64, 0, None, 0.0, 3, None, 0, None) == UNSUP


LSE = 0x60000000


def fwd_dv(lib, fn="mha_fwd_dv", q=Q, k=K, v=V, o=O, lse=None, B=2, H=3, Lq=64, Lk=64, d_k=64,
           d_v=64, mask=0, lens=None, scale=0.0):
    return getattr(lib, fn)(q, k, v, o, lse, B, H, Lq, Lk, d_k, d_v, mask, lens, scale, None)


@pytest.mark.parametrize("fn", ["mha_fwd_dv", "mha_fwd_f32_dv"])
def test_dv_entry_errors(lib, fn):
    assert fwd_dv(lib, fn, d_v=0) == SHAPE
    assert fwd_dv(lib, fn, d_v=-8) == SHAPE
    assert fwd_dv(lib, fn, mask=3) == MASK
    assert fwd_dv(lib, fn, lse=LSE + 2) == UNSUP
    assert fwd_dv(lib, fn, lse=Q) == ALIAS
    # out is [B, Lq, H, d_v]: with d_v = 128 it reaches 2*64*3*128 elements past O
    elem = 2 if fn == "mha_fwd_dv" else 4
    assert fwd_dv(lib, fn, d_v=128, o=V - 2 * 64 * 3 * 128 * elem + 64) == ALIAS
    assert fwd_dv(lib, fn, B=0) == OK


def test_dv_width_limits(lib):
    assert fwd_dv(lib, d_v=12) == UNSUP       # bf16: multiples of 8 ...
    assert fwd_dv(lib, d_v=264) == UNSUP      # ... up to 256
    assert fwd_dv(lib, d_k=20) == UNSUP
    assert fwd_dv(lib, fn="mha_fwd_f32_dv", d_v=257) == UNSUP


@pytest.mark.parametrize("fn", ["mha_fwd_lse", "mha_fwd_f32_lse"])
def test_lse_entry_errors(lib, fn):
    def call(lse=LSE, o=O, B=2, H=3, Lq=64, Lk=64, d=64, mask=0):
        return getattr(lib, fn)(Q, K, V, o, lse, B, H, Lq, Lk, d, mask, None, 0.0, None)
    assert call(lse=None) == NULL
    assert call(lse=LSE + 2) == UNSUP          # float32 lse needs 4-byte alignment
    assert call(lse=O + 64) == ALIAS           # lse overlaps out
    assert call(lse=Q) == ALIAS                # lse overlaps q
    assert call(o=None) == NULL                # the base checks still come first
    assert call(mask=1, Lk=65) == SHAPE
    assert call(B=0, lse=None) == OK           # empty query side: nothing to store


WS = 0x70000000
LENS_D = 0x78000000


def dec(lib, q=Q, k=K, v=V, o=O, lse=None, B=2, H=3, Lk=64, d=64, lens=LENS_D, scale=0.0,
        ws=None, ws_bytes=0):
    return lib.mha_decode(q, k, v, o, lse, B, H, Lk, d, lens, scale, ws, ws_bytes, None)


def test_decode_entry_errors(lib):
    assert dec(lib, B=-1) == SHAPE
    assert dec(lib, Lk=-1) == SHAPE
    assert dec(lib, d=100) == UNSUP                        # multiples of 8 up to 256
    assert dec(lib, d=264) == UNSUP
    assert dec(lib, scale=math.nan) == SCALE
    assert dec(lib, q=None) == NULL
    assert dec(lib, k=None) == NULL
    assert dec(lib, lens=None) == MASK                     # cache lengths are required
    assert dec(lib, q=Q + 8) == UNSUP
    assert dec(lib, lse=0x60000002) == UNSUP
    assert dec(lib, o=Q) == ALIAS
    assert dec(lib, lse=O) == ALIAS
    assert dec(lib, B=0) == OK and dec(lib, H=0, q=None) == OK
    # a small batch over a long cache is split: it needs the workspace
    need = lib.mha_decode_workspace_bytes(1, 4, 8192, 128)
    assert need > 0
    assert dec(lib, B=1, H=4, Lk=8192, d=128) == WORKSPACE
    assert dec(lib, B=1, H=4, Lk=8192, d=128, ws=WS, ws_bytes=need - 1) == WORKSPACE
    assert dec(lib, B=1, H=4, Lk=8192, d=128, ws=WS + 4, ws_bytes=need) == WORKSPACE
    # many heads over a short cache run in one pass and need none
    assert lib.mha_decode_workspace_bytes(64, 16, 256, 64) == 0
    assert lib.mha_decode_workspace_bytes(2, 3, 64, 96) == 0


DOUT, DQ, DK, DVG = 0x80000000, 0x90000000, 0xA0000000, 0xB0000000


def bwd(lib, d=64, mask=0, lens=None, lse=LSE, ws=WS, ws_bytes=1 << 20, out=O, dk=DK):
    return lib.mha_bwd(Q, K, V, out, DOUT, lse, DQ, dk, DVG, 2, 3, 64, 64, d, mask, lens, 0.0, ws,
                       ws_bytes, None)


def test_bwd_entry_errors(lib):
    assert bwd(lib, d=12) == UNSUP            # multiples of 8 up to 128
    assert bwd(lib, d=136) == UNSUP
    assert bwd(lib, mask=4) == MASK
    assert bwd(lib, mask=3) == MASK           # both masks need key_lens
    assert bwd(lib, lse=None) == NULL
    assert bwd(lib, ws=None) == WORKSPACE
    assert bwd(lib, out=O + 8) == UNSUP       # out and dk/dv are read / written by TMA
    assert bwd(lib, dk=DK + 8) == UNSUP
    assert bwd(lib, ws=Q) == ALIAS            # the workspace overlaps an input
    assert bwd(lib, ws=DQ + 256) == ALIAS     # ... or a gradient
    assert lib.mha_bwd_workspace_bytes(2, 3, 64, 64, 96) > 0
    assert lib.mha_bwd_workspace_bytes(2, 3, 64, 64, 12) == 0


XL, ML, WQ, WO, YL = 0x100000000, 0x110000000, 0x120000000, 0x130000000, 0x140000000
WSL = 0x150000000


def layer(lib, x=XL, mem=None, wq=WQ, wo=WO, y=YL, B=2, Lq=64, Lk=64, dm=512, H=8, dk=64,
          mask=0, lens=None, scale=0.0, ws=WSL, wsb=None):
    if wsb is None:
        wsb = lib.mha_layer_workspace_bytes(B, Lq, Lk, dm, H, dk)
    return lib.mha_layer_fwd(x, mem, wq, wo, y, B, Lq, Lk, dm, H, dk, mask, lens, scale, ws, wsb,
                             None)


def test_layer_entry_errors(lib):
    # every call below fails its checks before any device is touched
    assert layer(lib, B=-1) == SHAPE
    assert layer(lib, dm=0) == SHAPE
    assert layer(lib, Lk=65) == SHAPE                  # self-attention: Lk == Lq
    assert layer(lib, mem=ML, mask=1, Lk=65) == SHAPE  # causal: Lq == Lk
    assert layer(lib, mask=4) == MASK
    assert layer(lib, mask=2) == MASK                  # key padding needs key_lens
    assert layer(lib, scale=math.nan) == SCALE
    assert layer(lib, dk=12) == UNSUP
    assert layer(lib, dm=100) == UNSUP                 # d_model a multiple of 8
    assert layer(lib, x=XL + 8) == UNSUP
    assert layer(lib, x=None) == NULL
    assert layer(lib, wo=None) == NULL
    assert layer(lib, ws=None) == WORKSPACE
    assert layer(lib, ws=WSL + 16) == WORKSPACE
    assert layer(lib, wsb=1024) == WORKSPACE
    assert layer(lib, y=XL + 64) == ALIAS              # y overlaps x
    assert layer(lib, ws=WQ) == ALIAS                  # workspace overlaps the weights
    assert layer(lib, B=0) == OK
    # the Q|K|V projections and the heads' output, bf16: (3 + 1) x 2 x 64 x 512 x 2 bytes
    assert lib.mha_layer_workspace_bytes(2, 64, 64, 512, 8, 64) == 4 * 2 * 64 * 512 * 2
    assert lib.mha_layer_workspace_bytes(2, 64, 64, 512, 8, 12) == 0


AG, BG, CG = 0x160000000, 0x170000000, 0x180000000


def test_gemm_entry_errors(lib):
    f = lib.mha_gemm_bf16
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_longlong] * 3 + [ctypes.c_void_p]
    assert f(AG, BG, CG, -1, 8, 8, 8, 8, 8, None) == SHAPE
    assert f(AG, BG, CG, 8, 8, 16, 8, 8, 8, None) == SHAPE       # lda < K
    assert f(AG, BG, CG, 8, 16, 8, 8, 8, 16, None) == SHAPE      # ldb < N
    assert f(None, BG, CG, 8, 8, 8, 8, 8, 8, None) == NULL
    assert f(AG, BG, CG, 8, 8, 12, 12, 8, 8, None) == UNSUP      # rows not a multiple of 8
    assert f(AG + 8, BG, CG, 8, 8, 8, 8, 8, 8, None) == UNSUP    # base not 16-byte aligned
    assert f(AG, BG, AG + 16, 8, 8, 8, 8, 8, 8, None) == ALIAS   # c overlaps a
    assert f(AG, BG, CG, 0, 8, 8, 8, 8, 8, None) == OK           # nothing to compute
