"""GB300-native multi-head scaled dot-product attention forward.

``mha_fwd`` / ``mha_fwd_f32`` compute softmax(Q K^T * scale) V over every
sequence and head of [B, L, H, d_k] tensors ("Attention Is All You Need",
Section 3.2.1, Equation (1), applied to all heads in parallel as in
Section 3.2.2) with hand-written sm_103a CUDA kernels behind the C ABI of
``libmha.so`` (declared in ``include/mha.h``).  This package is the thin
Python binding: it marshals arguments and raises when the library is missing.
"""
from .inputs import (MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE, WORKLOADS, BY_NAME,
                     Workload, generate)

__all__ = ["MASK_NONE", "MASK_CAUSAL", "MASK_KEY_PADDING", "WORKLOADS", "BY_NAME",
           "Workload", "generate", "mha_fwd", "mha_fwd_f32", "mha_sync_status",
           "mha_status_string", "MhaError"]


def __getattr__(name):
    # The binding loads libmha.so on first use, so importing the package (for
    # the input generator, say) works on a machine without a GPU.
    if name in ("mha_fwd", "mha_fwd_f32", "mha_sync_status", "mha_status_string",
                "MhaError", "lib", "library_path"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
