"""Helpers for GPU-vs-oracle parity tests.

Tolerances (fixed by the target specification of this library):
  - float32 inputs, float32 arithmetic: max |O - O_ref| <= 1e-5;
  - bf16 inputs, float32 accumulation, bf16 output: max |O - O_ref| <= 1e-2
    and ||O - O_ref||_F / ||O_ref||_F <= 5e-3,
where O_ref is the float64 oracle evaluated on the exact float64 images of the
values the GPU received.

Row log-sum-exps (natural log, float32 on the GPU) are compared with
    |lse - lse_ref| <= 5e-4 + 1e-6 |lse_ref|,   and -inf exactly where the oracle has -inf.
Derivation: the row maximum comes from float32 scores whose tensor-core
accumulation over d_k <= 128 bf16 products errs by at most about
d_k * 2^-24 * sum|q_i k_i| * scale (about 1e-5 on the workloads, a few 1e-4 on
peaked rows with scale 1), and log(l) from a float32 sum of at most 4096
positive terms (relative error <= 4096 * 2^-24 = 2.4e-4 even in the worst
order) of exponentials with relative error about 2^-22.  A wrong log base, a
dropped maximum or a missing ln 2 errs by far more.

Outside the workloads' input distribution (nearly one-hot softmax rows with
|O| of several units) the bf16 rounding floor alone exceeds 1e-2: the kernel
rounds every probability p and every output to bf16 (unit roundoff 2^-8), so
an output row close to one value row carries up to 2^-8|O| from P and 2^-8|O|
from the final rounding.  Such cases use, element by element,
    |O - O_ref| <= 1e-2 + 2^-7 |O_ref|
together with the same relative Frobenius bound.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

BF16_MAX_ABS = 1e-2
BF16_REL_FRO = 5e-3
F32_MAX_ABS = 1e-5


def to_cuda(case):
    out = {}
    for name in ("q", "k", "v"):
        out[name] = case[name].cuda()
    out["key_lens"] = case["key_lens"].cuda() if case.get("key_lens") is not None else None
    return out


def gpu_run(binding, case, mask_kind, scale=0.0):
    g = to_cuda(case)
    fn = binding.mha_fwd if case["q"].dtype == torch.bfloat16 else binding.mha_fwd_f32
    o = fn(g["q"], g["k"], g["v"], mask_kind=mask_kind, key_lens=g["key_lens"], scale=scale)
    assert binding.mha_sync_status() == 0
    return o


def oracle_run(case, mask_kind, scale=None, return_lse=False):
    lens = case.get("key_lens")
    return oracle.mha(case["q"], case["k"], case["v"], mask_kind,
                      key_lens=lens.numpy() if lens is not None else None, scale=scale,
                      return_lse=return_lse)


def gpu_run_lse(binding, case, mask_kind, scale=0.0):
    g = to_cuda(case)
    fn = binding.mha_fwd if case["q"].dtype == torch.bfloat16 else binding.mha_fwd_f32
    o, lse = fn(g["q"], g["k"], g["v"], mask_kind=mask_kind, key_lens=g["key_lens"],
                scale=scale, return_lse=True)
    assert binding.mha_sync_status() == 0
    return o, lse


# Gradient (mha_bwd), relative to the reference's Frobenius norm and largest
# magnitude.  The inputs are exact in both; the kernel rounds three things to
# bf16 (unit roundoff u = 2^-9): the weights P before dV = P^T dO, dS before
# dK = dS^T Q and dQ = dS K, and the gradients themselves.  Each adds a
# random relative error of about u / sqrt(3) per element, about u in all
# (measured 1.7e-3 .. 3.1e-3 Frobenius, <= 5.4e-3 largest).  The Frobenius
# bound is the forward's bf16 one, 5e-3 (about 2.6u); the largest element
# may err by 8u.  A dropped D, a lost scale or a transposed operand errs by
# O(1).
BWD_REL_FRO = 5e-3
BWD_REL_MAX = 8 * 2.0 ** -9

LSE_ABS = 5e-4
LSE_REL = 1e-6


def assert_lse_close(lse, ref, what=""):
    got = lse.detach().to("cpu", torch.float64).numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{what}: -inf rows differ"
    assert np.all(np.isfinite(got[~inf_ref])), f"{what}: non-finite lse"
    err = np.abs(got[~inf_ref] - ref[~inf_ref])
    bound = LSE_ABS + LSE_REL * np.abs(ref[~inf_ref])
    worst = float((err - bound).max()) if err.size else -1.0
    assert worst <= 0, f"{what}: lse error exceeds 5e-4 + 1e-6|lse| by {worst:.3e} (max err {err.max():.3e})"


def errors(out, ref):
    o = out.detach().to("cpu", torch.float64).numpy()
    diff = o - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    ref_norm = float(np.linalg.norm(ref))
    rel_fro = float(np.linalg.norm(diff) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(diff))
    return max_abs, rel_fro


def assert_bf16_close(out, ref, what=""):
    assert torch.isfinite(out.float()).all(), f"{what}: non-finite output"
    max_abs, rel = errors(out, ref)
    assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_FRO, \
        f"{what}: max_abs {max_abs:.3e} (<= {BF16_MAX_ABS}), rel_fro {rel:.3e} (<= {BF16_REL_FRO})"
    return max_abs, rel


def assert_bf16_close_rounding_aware(out, ref, what=""):
    assert torch.isfinite(out.float()).all(), f"{what}: non-finite output"
    o = out.detach().to("cpu", torch.float64).numpy()
    excess = np.abs(o - ref) - (BF16_MAX_ABS + 2.0 ** -7 * np.abs(ref))
    _, rel = errors(out, ref)
    assert excess.max() <= 0 and rel <= BF16_REL_FRO, \
        f"{what}: worst excess over 1e-2 + 2^-7|ref| is {excess.max():.3e}, rel_fro {rel:.3e}"
    return float(excess.max()), rel


def assert_f32_close(out, ref, what=""):
    max_abs, rel = errors(out, ref)
    assert max_abs <= F32_MAX_ABS, f"{what}: max_abs {max_abs:.3e} (<= {F32_MAX_ABS})"
    return max_abs, rel


# The multi-head layer (mha_layer_fwd) against the float64 layer oracle on the
# same bf16 inputs and weights, relative to the reference's Frobenius norm and
# largest magnitude.  Beyond the attention's own roundings (P and O to bf16)
# the layer rounds the Q, K, V projections and the output y to bf16: five
# roundings of unit roundoff u = 2^-9 on the path, each a random relative
# error of about u / sqrt(3) per element (Q and K errors reach y through the
# scores, scaled by |s| ~ 1 on these Xavier-scaled inputs), about 1.3u in all;
# the bounds allow 4u (Frobenius) and 8u (largest element).  A wrong head
# slice, a swapped K/V block or a dropped scale errs by O(1).
LAYER_REL_FRO = 4 * 2.0 ** -9
LAYER_REL_MAX = 8 * 2.0 ** -9


def assert_layer_close(y, ref, what=""):
    g = y.to(torch.float64).numpy() if hasattr(y, "numpy") else np.asarray(y, dtype=np.float64)
    scale = float(np.abs(ref).max()) or 1.0
    fro = float(np.linalg.norm(ref)) or 1.0
    rel_max = float(np.abs(g - ref).max()) / scale
    rel_fro = float(np.linalg.norm(g - ref)) / fro
    assert rel_fro <= LAYER_REL_FRO and rel_max <= LAYER_REL_MAX, \
        f"{what}: relative Frobenius {rel_fro:.3e} (bound {LAYER_REL_FRO:.3e}), " \
        f"relative max {rel_max:.3e} (bound {LAYER_REL_MAX:.3e})"
    return rel_fro, rel_max
