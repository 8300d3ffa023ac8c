"""Float64 CPU oracle for multi-head scaled dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package.  It shares no code
with the CUDA library (``transformer_head_scaled_sdpa_gb300``) and imports
nothing from it; the product path never calls it.

The arithmetic lives in ``mha_oracle.c`` (plain C, float64, one query row at a
time): score s_j = scale * q.k_j, weights a_j = e^{s_j} / sum_i e^{s_i},
output o = sum_j a_j v_j ("Attention Is All You Need", Section 3.2.1,
Equation (1); formula page transformer-attention, section 証明), with the
causal and key-padding masks removing keys before the softmax.  This module
compiles that file with gcc, loads it with ctypes and marshals arrays; its one
piece of arithmetic of its own is ``mha_layer``: the multi-head layer of
Section 3.2.2 as float64 matrix products (numpy) around that attention.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(the pages' worked examples, closed-form invariants, brute force on tiny
inputs and a library cross-check).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KEY_PADDING = 2
MASK_CAUSAL_KEY_PADDING = 3  # both masks (a decoder over padded sequences)

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mha_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_default = None


def compile_source(src: str, out_path: str) -> str:
    """gcc a C source of the oracle into a shared library at ``out_path``."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-std=c11", "-Wall", "-shared", "-fPIC",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``mha_oracle.c`` into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE))
    if force or not fresh:
        compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _as_f64(x) -> np.ndarray:
    """Exact float64 image of a numpy array or a (CPU) torch tensor."""
    if hasattr(x, "detach"):  # torch tensor: widen on the torch side (exact)
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_mha_f64.restype = ctypes.c_int
        lib.oracle_mha_f64.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double,
            ctypes.c_int]
        lib.oracle_mha_dv_f64.restype = ctypes.c_int
        lib.oracle_mha_dv_f64.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double,
            ctypes.c_int]
        lib.oracle_mha_bwd_f64.restype = ctypes.c_int
        lib.oracle_mha_bwd_f64.argtypes = [ctypes.c_void_p] * 7 + [
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double,
            ctypes.c_int]
        lib.oracle_default_threads.restype = ctypes.c_int
        lib.oracle_default_threads.argtypes = []
        self.lib = lib

    def default_threads(self) -> int:
        return int(self.lib.oracle_default_threads())

    def mha(self, q, k, v, mask_kind: int = MASK_NONE, key_lens=None, scale=None,
            threads: int | None = None, return_lse: bool = False):
        """Attention over all heads: q [B,Lq,H,d_k], k [B,Lk,H,d_k] and v
        [B,Lk,H,d_v] -> o [B,Lq,H,d_v] (d_v may differ from d_k).

        ``scale`` None means 1/sqrt(d_k).  ``key_lens`` ([B] integers) is read
        only when the mask includes key padding (``MASK_KEY_PADDING``,
        ``MASK_CAUSAL_KEY_PADDING``).  With ``return_lse`` also returns the row
        log-sum-exp of the scaled scores, shape [B, H, Lq].
        """
        q = _as_f64(q)
        k = _as_f64(k)
        v = _as_f64(v)
        if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
            raise ValueError("q, k, v must be [B, L, H, d]")
        B, Lq, H, d = q.shape
        Lk = k.shape[1]
        d_v = v.shape[3]
        if k.shape != (B, Lk, H, d) or v.shape != (B, Lk, H, d_v):
            raise ValueError("k must be [B, Lk, H, d_k] and v [B, Lk, H, d_v] matching q")
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        lens = None
        if int(mask_kind) & MASK_KEY_PADDING:
            if key_lens is None:
                raise ValueError("key padding needs key_lens")
            if hasattr(key_lens, "detach"):
                key_lens = key_lens.detach().cpu().numpy()
            lens = np.ascontiguousarray(np.asarray(key_lens, dtype=np.int32))
            if lens.shape != (B,):
                raise ValueError("key_lens must have shape [B]")
        out = np.empty((B, Lq, H, d_v), dtype=np.float64)
        lse = np.empty((B, H, Lq), dtype=np.float64) if return_lse else None
        rc = self.lib.oracle_mha_dv_f64(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data,
            lse.ctypes.data if lse is not None else None,
            B, H, Lq, Lk, d, d_v, int(mask_kind),
            lens.ctypes.data if lens is not None else None,
            float(scale), int(threads) if threads else 0)
        if rc != 0:
            raise ValueError(f"oracle_mha_dv_f64 rejected its arguments (code {rc})")
        return (out, lse) if return_lse else out


    def mha_bwd(self, q, k, v, dout, mask_kind: int = MASK_NONE, key_lens=None, scale=None,
                threads: int | None = None):
        """Gradient of attention for a loss with dL/dout = ``dout``
        ([B,Lq,H,d]): returns (dq, dk, dv) in the layouts of q, k, v."""
        q, k, v, dout = (_as_f64(x) for x in (q, k, v, dout))
        if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
            raise ValueError("q, k, v must be [B, L, H, d]")
        B, Lq, H, d = q.shape
        Lk = k.shape[1]
        if k.shape != (B, Lk, H, d) or v.shape != (B, Lk, H, d) or dout.shape != q.shape:
            raise ValueError("shapes do not match")
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        lens = None
        if int(mask_kind) & MASK_KEY_PADDING:
            if key_lens is None:
                raise ValueError("key padding needs key_lens")
            if hasattr(key_lens, "detach"):
                key_lens = key_lens.detach().cpu().numpy()
            lens = np.ascontiguousarray(np.asarray(key_lens, dtype=np.int32))
        dq = np.empty_like(q)
        dk = np.empty_like(k)
        dv = np.empty_like(v)
        rc = self.lib.oracle_mha_bwd_f64(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
            dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, B, H, Lq, Lk, d, int(mask_kind),
            lens.ctypes.data if lens is not None else None, float(scale),
            int(threads) if threads else 0)
        if rc != 0:
            raise ValueError(f"oracle_mha_bwd_f64 rejected its arguments (code {rc})")
        return dq, dk, dv


def _get() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def mha_bwd(q, k, v, dout, mask_kind: int = MASK_NONE, key_lens=None, scale=None,
            threads: int | None = None):
    """Module-level convenience over the default oracle build (see Oracle.mha_bwd)."""
    return _get().mha_bwd(q, k, v, dout, mask_kind, key_lens, scale, threads)


def default_threads() -> int:
    """Threads the oracle uses when ``threads`` is not given."""
    return _get().default_threads()


def mha(q, k, v, mask_kind: int = MASK_NONE, key_lens=None, scale=None,
        threads: int | None = None, return_lse: bool = False):
    """Attention over all heads with the default build (see ``Oracle.mha``)."""
    return _get().mha(q, k, v, mask_kind=mask_kind, key_lens=key_lens, scale=scale,
                      threads=threads, return_lse=return_lse)


def mha_layer(x, w_qkv, w_o, H: int, mem=None, mask_kind: int = MASK_NONE, key_lens=None,
              scale=None, threads: int | None = None):
    """The multi-head attention layer ("Attention Is All You Need", Section
    3.2.2): MultiHead(Q, K, V) = Concat(head_1, ..., head_H) W^O with
    head_h = Attention(Q W_h^Q, K W_h^K, V W_h^V), queries from x [B, Lq,
    d_model] and keys and values from ``mem`` [B, Lk, d_model] (x itself when
    None: self-attention).  w_qkv [d_model, 3 H d_k] holds W^Q, W^K, W^V side by
    side, head h at columns h d_k .. h d_k + d_k - 1 of each; w_o [H d_k,
    d_model].  All float64: the three projections, the attention of the C
    oracle over all heads, then the output projection of the heads'
    concatenation.  Returns y [B, Lq, d_model]."""
    x = _as_f64(x)
    mem = x if mem is None else _as_f64(mem)
    w_qkv = _as_f64(w_qkv)
    w_o = _as_f64(w_o)
    B, Lq, d_model = x.shape
    Lk = mem.shape[1]
    hd = w_qkv.shape[1] // 3
    if w_qkv.shape != (d_model, 3 * hd) or hd % H != 0 or w_o.shape != (hd, d_model):
        raise ValueError("w_qkv must be [d_model, 3 H d_k] and w_o [H d_k, d_model]")
    if mem.shape != (B, Lk, d_model):
        raise ValueError("mem must be [B, Lk, d_model]")
    d_k = hd // H
    q = (x @ w_qkv[:, :hd]).reshape(B, Lq, H, d_k)
    k = (mem @ w_qkv[:, hd:2 * hd]).reshape(B, Lk, H, d_k)
    v = (mem @ w_qkv[:, 2 * hd:]).reshape(B, Lk, H, d_k)
    o = mha(q, k, v, mask_kind, key_lens=key_lens, scale=scale, threads=threads)
    return o.reshape(B, Lq, hd) @ w_o
