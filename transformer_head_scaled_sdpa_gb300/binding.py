"""ctypes binding of libmha.so (C ABI in ``include/mha.h``).

Argument marshalling only: every step of the attention forward runs in the
library's CUDA kernels.  Tensors are torch tensors (device memory and streams
come from PyTorch); their shapes are [B, L, H, d_k].  If the library has not
been built, or cannot be loaded, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MHA_OK = 0
STATUS_NAMES = {
    0: "MHA_OK", 1: "MHA_ERR_NULL", 2: "MHA_ERR_SHAPE", 3: "MHA_ERR_UNSUPPORTED",
    4: "MHA_ERR_MASK", 5: "MHA_ERR_SCALE", 6: "MHA_ERR_LAUNCH", 7: "MHA_ERR_TIMEOUT",
    8: "MHA_ERR_ALIAS", 9: "MHA_ERR_WORKSPACE",
}

_lock = threading.Lock()
_lib = None

_c_p = ctypes.c_void_p
_c_i = ctypes.c_int
_FWD_ARGS = [_c_p, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_p,
             ctypes.c_float, _c_p]
_FWD_LSE_ARGS = _FWD_ARGS[:4] + [_c_p] + _FWD_ARGS[4:]


class MhaError(RuntimeError):
    """A non-zero mha_status from the library."""

    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.code, self.code)} "
                         f"({mha_status_string(self.code)})")


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded libmha.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it first "
                    "(python -m transformer_head_scaled_sdpa_gb300.build)")
            h = ctypes.CDLL(path)
            h.mha_fwd.restype = _c_i
            h.mha_fwd.argtypes = _FWD_ARGS
            h.mha_fwd_f32.restype = _c_i
            h.mha_fwd_f32.argtypes = _FWD_ARGS
            h.mha_fwd_lse.restype = _c_i
            h.mha_fwd_lse.argtypes = _FWD_LSE_ARGS
            h.mha_fwd_f32_lse.restype = _c_i
            h.mha_fwd_f32_lse.argtypes = _FWD_LSE_ARGS
            h.mha_layer_fwd.restype = _c_i
            h.mha_layer_fwd.argtypes = [_c_p] * 5 + [_c_i] * 7 + [_c_p, ctypes.c_float, _c_p,
                                                                   ctypes.c_size_t, _c_p]
            h.mha_layer_workspace_bytes.restype = ctypes.c_size_t
            h.mha_layer_workspace_bytes.argtypes = [_c_i] * 6
            h.mha_gemm_bf16.restype = _c_i
            h.mha_gemm_bf16.argtypes = [_c_p] * 3 + [_c_i] * 3 + [ctypes.c_longlong] * 3 + [_c_p]
            for name in ("mha_fwd_dv", "mha_fwd_f32_dv"):
                getattr(h, name).restype = _c_i
                getattr(h, name).argtypes = [_c_p] * 5 + [_c_i] * 7 + [_c_p, ctypes.c_float, _c_p]
            h.mha_bwd.restype = _c_i
            h.mha_bwd.argtypes = [_c_p] * 9 + [_c_i] * 6 + [_c_p, ctypes.c_float, _c_p,
                                                            ctypes.c_size_t, _c_p]
            h.mha_bwd_workspace_bytes.restype = ctypes.c_size_t
            h.mha_bwd_workspace_bytes.argtypes = [_c_i] * 5
            h.mha_decode.restype = _c_i
            h.mha_decode.argtypes = [_c_p] * 5 + [_c_i] * 4 + [_c_p, ctypes.c_float, _c_p,
                                                               ctypes.c_size_t, _c_p]
            h.mha_decode_static.restype = _c_i
            h.mha_decode_static.argtypes = [_c_p] * 5 + [_c_i] * 4 + [_c_p, ctypes.c_float, _c_p]
            h.mha_decode_static_scratch_bytes.restype = ctypes.c_size_t
            h.mha_decode_static_scratch_bytes.argtypes = []
            h.mha_decode_workspace_bytes.restype = ctypes.c_size_t
            h.mha_decode_workspace_bytes.argtypes = [_c_i] * 4
            h.mha_fwd_host_workspace_bytes.restype = ctypes.c_size_t
            h.mha_fwd_host_workspace_bytes.argtypes = [_c_i] * 6
            h.mha_fwd_host.restype = _c_i
            h.mha_fwd_host.argtypes = _FWD_ARGS[:-1] + [_c_i, _c_p, ctypes.c_size_t, _c_p]
            h.mha_selftest_timeout.restype = _c_i
            h.mha_selftest_timeout.argtypes = [_c_p]
            h.mha_debug_withhold_p.restype = None
            h.mha_debug_withhold_p.argtypes = [_c_i]
            h.mha_sync_status.restype = _c_i
            h.mha_sync_status.argtypes = [_c_p]
            h.mha_status_string.restype = ctypes.c_char_p
            h.mha_status_string.argtypes = [_c_i]
            h.mha_last_launch_info.restype = None
            h.mha_last_launch_info.argtypes = [ctypes.POINTER(_c_i)] * 4
            _lib = h
    return _lib


def mha_status_string(code: int) -> str:
    return lib().mha_status_string(int(code)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _shape(q, k, v, allow_dv=False):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, L, H, d_k]")
    B, Lq, H, d = q.shape
    Lk = k.shape[1]
    d_v = v.shape[3] if allow_dv else d
    if tuple(k.shape) != (B, Lk, H, d) or tuple(v.shape) != (B, Lk, H, d_v):
        raise ValueError(f"k {tuple(k.shape)} / v {tuple(v.shape)} do not match q {tuple(q.shape)}")
    return B, H, Lq, Lk, d


def _check_tensor(t, name, dtype, device_kind):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device.type != device_kind:
        raise ValueError(f"{name} must be on {device_kind}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _call_fwd(fn_name, dtype, q, k, v, out, mask_kind, key_lens, scale, stream,
              lse=None, want_lse=False):
    B, H, Lq, Lk, d = _shape(q, k, v, allow_dv=True)
    d_v = v.shape[3]
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, dtype, "cuda")
    if out is None:
        out = torch.empty((B, Lq, H, d_v), dtype=dtype, device=q.device)
    _check_tensor(out, "out", dtype, "cuda")
    if tuple(out.shape) != (B, Lq, H, d_v):
        raise ValueError("out must be [B, Lq, H, d_v]")
    lens_ptr = None
    if key_lens is not None:
        _check_tensor(key_lens, "key_lens", torch.int32, "cuda")
        if tuple(key_lens.shape) != (B,):
            raise ValueError("key_lens must be [B]")
        lens_ptr = key_lens.data_ptr()
    if d_v != d:
        # value rows of their own width: the *_dv entry (lse optional)
        if want_lse:
            if lse is None:
                lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
            _check_tensor(lse, "lse", torch.float32, "cuda")
            if tuple(lse.shape) != (B, H, Lq):
                raise ValueError("lse must be [B, H, Lq]")
        fn_name += "_dv"
        rc = getattr(lib(), fn_name)(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                     lse.data_ptr() if want_lse else None, B, H, Lq, Lk, d, d_v,
                                     int(mask_kind), lens_ptr, float(scale),
                                     _stream_handle(stream))
        if rc != MHA_OK:
            raise MhaError(rc, fn_name)
        return (out, lse) if want_lse else out
    if not want_lse:
        rc = getattr(lib(), fn_name)(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                     B, H, Lq, Lk, d, int(mask_kind), lens_ptr, float(scale),
                                     _stream_handle(stream))
        if rc != MHA_OK:
            raise MhaError(rc, fn_name)
        return out
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    _check_tensor(lse, "lse", torch.float32, "cuda")
    if tuple(lse.shape) != (B, H, Lq):
        raise ValueError("lse must be [B, H, Lq]")
    fn_name += "_lse"
    rc = getattr(lib(), fn_name)(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr(), B, H, Lq, Lk, d, int(mask_kind), lens_ptr,
                                 float(scale), _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, fn_name)
    return out, lse


def mha_fwd(q, k, v, out=None, mask_kind: int = 0, key_lens=None, scale: float = 0.0,
            stream=None, return_lse: bool = False, lse=None):
    """bf16 attention forward on the GPU (tcgen05 kernel); returns ``out``, or
    ``(out, lse)`` with ``return_lse`` (lse: float32 [B, H, Lq], natural log).
    v (and out) may have a width d_v of their own: q, k [.., d_k], v [.., d_v]."""
    return _call_fwd("mha_fwd", torch.bfloat16, q, k, v, out, mask_kind, key_lens, scale,
                     stream, lse, return_lse)


def mha_fwd_f32(q, k, v, out=None, mask_kind: int = 0, key_lens=None, scale: float = 0.0,
                stream=None, return_lse: bool = False, lse=None):
    """float32 attention forward on the GPU (SIMT kernel); returns ``out``, or
    ``(out, lse)`` with ``return_lse``."""
    return _call_fwd("mha_fwd_f32", torch.float32, q, k, v, out, mask_kind, key_lens, scale,
                     stream, lse, return_lse)


def mha_bwd(q, k, v, out, dout, lse, mask_kind: int = 0, key_lens=None, scale: float = 0.0,
            dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradient of mha_fwd (bf16): returns (dq, dk, dv) for dL/dout = ``dout``,
    given the forward's ``out`` and ``lse`` (from mha_fwd(..., return_lse=True))."""
    B, H, Lq, Lk, d = _shape(q, k, v)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _check_tensor(t, n, torch.bfloat16, "cuda")
    if tuple(out.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("out and dout must have q's shape")
    _check_tensor(lse, "lse", torch.float32, "cuda")
    if tuple(lse.shape) != (B, H, Lq):
        raise ValueError("lse must be [B, H, Lq]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, ref, n in ((dq, q, "dq"), (dk, k, "dk"), (dv, v, "dv")):
        _check_tensor(t, n, torch.bfloat16, "cuda")
        if tuple(t.shape) != tuple(ref.shape):
            raise ValueError(f"{n} must have the shape of its input")
    lens_ptr = None
    if key_lens is not None:
        _check_tensor(key_lens, "key_lens", torch.int32, "cuda")
        lens_ptr = key_lens.data_ptr()
    need = int(lib().mha_bwd_workspace_bytes(B, H, Lq, Lk, d))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check_tensor(workspace, "workspace", torch.uint8, "cuda")
    rc = lib().mha_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                       dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                       dv.data_ptr(), B, H, Lq, Lk, d, int(mask_kind), lens_ptr, float(scale),
                       workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_bwd")
    return dq, dk, dv


def layer_workspace_bytes(B, Lq, Lk, d_model, H, d_k) -> int:
    return int(lib().mha_layer_workspace_bytes(B, Lq, Lk, d_model, H, d_k))


def mha_layer_fwd(x, w_qkv, w_o, H: int, mem=None, mask_kind: int = 0, key_lens=None,
                  scale: float = 0.0, y=None, workspace=None, stream=None):
    """One multi-head attention layer (bf16): y = Concat(heads) W^O with
    head_h = Attention(x W_h^Q, m W_h^K, m W_h^V), m = ``mem`` or x.
    x [B, Lq, d_model], mem [B, Lk, d_model] or None, w_qkv [d_model, 3 H d_k],
    w_o [H d_k, d_model]; returns y [B, Lq, d_model]."""
    if x.dim() != 3 or w_qkv.dim() != 2 or w_o.dim() != 2:
        raise ValueError("x must be [B, Lq, d_model], w_qkv and w_o matrices")
    B, Lq, d_model = x.shape
    hd3 = w_qkv.shape[1]
    if hd3 % (3 * H) != 0 or tuple(w_qkv.shape) != (d_model, hd3):
        raise ValueError("w_qkv must be [d_model, 3 H d_k]")
    d_k = hd3 // (3 * H)
    if tuple(w_o.shape) != (H * d_k, d_model):
        raise ValueError("w_o must be [H d_k, d_model]")
    Lk = Lq if mem is None else mem.shape[1]
    tensors = [(x, "x"), (w_qkv, "w_qkv"), (w_o, "w_o")]
    if mem is not None:
        if mem.dim() != 3 or mem.shape[0] != B or mem.shape[2] != d_model:
            raise ValueError("mem must be [B, Lk, d_model]")
        tensors.append((mem, "mem"))
    for t, n in tensors:
        _check_tensor(t, n, torch.bfloat16, "cuda")
    if y is None:
        y = torch.empty_like(x)
    _check_tensor(y, "y", torch.bfloat16, "cuda")
    if tuple(y.shape) != tuple(x.shape):
        raise ValueError("y must have x's shape")
    lens_ptr = None
    if key_lens is not None:
        _check_tensor(key_lens, "key_lens", torch.int32, "cuda")
        lens_ptr = key_lens.data_ptr()
    need = layer_workspace_bytes(B, Lq, Lk, d_model, H, d_k)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check_tensor(workspace, "workspace", torch.uint8, "cuda")
    rc = lib().mha_layer_fwd(x.data_ptr(), mem.data_ptr() if mem is not None else None,
                             w_qkv.data_ptr(), w_o.data_ptr(), y.data_ptr(), B, Lq, Lk, d_model,
                             H, d_k, int(mask_kind), lens_ptr, float(scale), workspace.data_ptr(),
                             workspace.numel(), _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_layer_fwd")
    return y


def mha_gemm_bf16(a, b, c=None, stream=None):
    """c = a @ b on the library's tensor-core GEMM: a [M, K], b [K, N] bf16
    CUDA matrices whose rows may be strided (stride(1) == 1, stride(0) a
    multiple of 8 elements, e.g. column blocks of a wider matrix); c [M, N]
    (allocated when not given, else written in place, same row rules)."""
    for t, n in ((a, "a"), (b, "b")):
        if t.dim() != 2 or t.dtype != torch.bfloat16 or not t.is_cuda or t.stride(1) != 1:
            raise ValueError(f"{n} must be a row-major bf16 CUDA matrix")
    M, K = a.shape
    if b.shape[0] != K:
        raise ValueError(f"inner sizes differ: a {tuple(a.shape)}, b {tuple(b.shape)}")
    N = b.shape[1]
    if c is None:
        c = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    if c.dim() != 2 or tuple(c.shape) != (M, N) or c.dtype != torch.bfloat16 or c.stride(1) != 1:
        raise ValueError("c must be a row-major bf16 [M, N] matrix")
    rc = lib().mha_gemm_bf16(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                             max(a.stride(0), K), max(b.stride(0), N), max(c.stride(0), N),
                             _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_gemm_bf16")
    return c


def decode_workspace_bytes(B, H, Lk, d_k) -> int:
    return int(lib().mha_decode_workspace_bytes(B, H, Lk, d_k))


def mha_decode_static(q, k_cache, v_cache, cache_lens, out=None, scale: float = 0.0,
                      stream=None, return_lse: bool = False, lse=None):
    """mha_decode with the library's fixed device scratch instead of a
    workspace (calls on one device must not overlap in time)."""
    return mha_decode(q, k_cache, v_cache, cache_lens, out=out, scale=scale, stream=stream,
                      return_lse=return_lse, lse=lse, _static=True)


def mha_decode(q, k_cache, v_cache, cache_lens, out=None, scale: float = 0.0, workspace=None,
               stream=None, return_lse: bool = False, lse=None, _static: bool = False):
    """One decode step (bf16): q [B, H, d] (or [B, 1, H, d]) against the first
    cache_lens[b] rows of k_cache / v_cache [B, Lk, H, d].  Returns out
    [B, H, d] (q's shape), or (out, lse) with ``return_lse``.  ``workspace``
    (uint8 CUDA tensor) is allocated when not given."""
    if q.dim() == 4:
        if q.shape[1] != 1:
            raise ValueError("q must be [B, H, d] or [B, 1, H, d]")
    elif q.dim() != 3:
        raise ValueError("q must be [B, H, d] or [B, 1, H, d]")
    B, H, d = q.shape[0], q.shape[-2], q.shape[-1]
    if k_cache.dim() != 4 or tuple(k_cache.shape[::2]) != (B, H) or k_cache.shape[3] != d \
            or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError(f"caches {tuple(k_cache.shape)} / {tuple(v_cache.shape)} do not match q")
    Lk = k_cache.shape[1]
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_tensor(t, n, torch.bfloat16, "cuda")
    _check_tensor(cache_lens, "cache_lens", torch.int32, "cuda")
    if tuple(cache_lens.shape) != (B,):
        raise ValueError("cache_lens must be [B]")
    if out is None:
        out = torch.empty_like(q)
    _check_tensor(out, "out", torch.bfloat16, "cuda")
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    lse_ptr = None
    if return_lse:
        if lse is None:
            lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
        _check_tensor(lse, "lse", torch.float32, "cuda")
        if tuple(lse.shape) != (B, H):
            raise ValueError("lse must be [B, H]")
        lse_ptr = lse.data_ptr()
    if _static:
        rc = lib().mha_decode_static(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     out.data_ptr(), lse_ptr, B, H, Lk, d,
                                     cache_lens.data_ptr(), float(scale), _stream_handle(stream))
        if rc != MHA_OK:
            raise MhaError(rc, "mha_decode_static")
        return (out, lse) if return_lse else out
    need = decode_workspace_bytes(B, H, Lk, d)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _check_tensor(workspace, "workspace", torch.uint8, "cuda")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    rc = lib().mha_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                          lse_ptr, B, H, Lk, d, cache_lens.data_ptr(), float(scale), ws_ptr,
                          ws_bytes, _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_decode")
    return (out, lse) if return_lse else out


def host_workspace_bytes(B, H, Lq, Lk, d_k, elem_bytes) -> int:
    return int(lib().mha_fwd_host_workspace_bytes(B, H, Lq, Lk, d_k, elem_bytes))


def mha_fwd_host(q, k, v, out, workspace, mask_kind: int = 0, key_lens=None,
                 scale: float = 0.0, stream=None) -> int:
    """Attention on HOST tensors (pinned for async copies) through the C ABI's
    host-buffer entry: H2D copies, the kernel and the D2H copy of ``out`` all
    run on ``stream``; returns once ``out`` holds the result."""
    B, H, Lq, Lk, d = _shape(q, k, v)
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("host tensors must be bf16 or float32")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check_tensor(t, n, dtype, "cpu")
    lens_ptr = None
    if key_lens is not None:
        _check_tensor(key_lens, "key_lens", torch.int32, "cpu")
        lens_ptr = key_lens.data_ptr()
    _check_tensor(workspace, "workspace", torch.uint8, "cuda")
    rc = lib().mha_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            B, H, Lq, Lk, d, int(mask_kind), lens_ptr, float(scale),
                            2 if dtype == torch.bfloat16 else 4, workspace.data_ptr(),
                            workspace.numel(), _stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_fwd_host")
    return rc


def mha_sync_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device status code."""
    return int(lib().mha_sync_status(_stream_handle(stream)))


def mha_selftest_timeout(stream=None) -> int:
    """Launch the bounded-wait self-test kernel (see include/mha.h)."""
    rc = lib().mha_selftest_timeout(_stream_handle(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_selftest_timeout")
    return rc


def mha_debug_withhold_p(on: bool) -> None:
    """Test hook: make later mha_fwd launches run out a pipeline wait."""
    lib().mha_debug_withhold_p(1 if on else 0)


def last_launch_info() -> dict:
    vals = [ctypes.c_int(0) for _ in range(4)]
    lib().mha_last_launch_info(*[ctypes.byref(x) for x in vals])
    return dict(zip(("kernels", "grid", "block", "smem"), (x.value for x in vals)))
