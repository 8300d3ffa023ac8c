"""Plausible mistakes planted in copies of the oracle (on the CPU) must each
fail at least one pin, which shows the pins can tell a wrong oracle apart."""
import math
import os

import pytest

import oracle
from tests import oracle_bwd_pins, oracle_pins

# (name, text in mha_oracle.c, replacement)
C_MUTANTS = [
    ("scale_dropped", "s[j] = scale * dot;", "s[j] = dot;"),
    ("values_read_from_keys", "const double* v_row = v + j * v_row_stride;",
     "const double* v_row = k + j * k_row_stride;"),
    ("diagonal_masked", "n = i + 1 < Lk ? i + 1 : Lk;", "n = i < Lk ? i : Lk;"),
    ("causal_ignored", "n = i + 1 < Lk ? i + 1 : Lk;", "n = Lk;"),
    ("no_normalisation", "for (int64_t j = 0; j < n; ++j) s[j] /= sum;", ""),
    ("max_not_subtracted", "s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    ("head_offset_dropped", "k + (b * Lk * H + h) * d", "k + (b * Lk * H) * d"),
    ("row_order_wrong", "const int64_t h = (r / Lq) % H;", "const int64_t h = r % H;"),
    ("padding_length_off_by_one", "n = len;", "n = len > 0 ? len - 1 : 0;"),
    ("query_row_stride_wrong", "q + ((b * Lq + i) * H + h) * d", "q + ((b * Lq + h) * H + i) * d"),
    # both masks together: padding dropped whenever the causal bit is set
    ("combined_mask_padding_dropped", "if (len < n) n = len;",
     "if (len < n && !(mask_kind & ORACLE_MASK_CAUSAL)) n = len;"),
    # d_v != d_k: value rows or output rows laid out with the key width
    ("value_stride_uses_dk", "H * d_k, H * d_v, scale, s", "H * d_k, H * d_k, scale, s"),
    ("output_stride_uses_dk", "double* o_row = out + ((b * Lq + i) * H + h) * d_v;",
     "double* o_row = out + ((b * Lq + i) * H + h) * d_k;"),
]


def _run_checks(mha):
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mha)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name,old,new", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_c_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / f"{name}.c"
    mutated.write_text(src.replace(old, new), encoding="utf-8")
    lib = oracle.compile_source(str(mutated), str(tmp_path / f"lib{name}.so"))
    failed = _run_checks(oracle.Oracle(lib).mha)
    assert failed, f"mutant {name} passed every pin"


def test_default_scale_mutant_is_caught():
    """Reading the formula page's rendering literally (divide by d_k, not sqrt)."""
    base = oracle.Oracle(oracle.build())

    def mha_over_dk(q, k, v, mask_kind=0, key_lens=None, scale=None, threads=None,
                    return_lse=False):
        if scale is None:
            scale = 1.0 / q.shape[-1]
        return base.mha(q, k, v, mask_kind, key_lens, scale, threads, return_lse)

    assert _run_checks(mha_over_dk)


# planted in the gradient (oracle_mha_bwd_f64); the forward stays correct
BWD_MUTANTS = [
    ("bwd_jacobian_mean_dropped", "const double ds = a[j] * (g[j] - ag);", "const double ds = a[j] * g[j];"),
    ("bwd_jacobian_sign", "const double ds = a[j] * (g[j] - ag);", "const double ds = a[j] * (ag - g[j]);"),
    ("bwd_dq_scale_dropped", "dq_row[c] += scale * ds * k_bh[j * rs + c];", "dq_row[c] += ds * k_bh[j * rs + c];"),
    ("bwd_dv_from_ds", "dv_bh[j * rs + c] += a[j] * do_row[c];", "dv_bh[j * rs + c] += ds * do_row[c];"),
    ("bwd_dk_from_keys", "dk_bh[j * rs + c] += scale * ds * q_row[c];", "dk_bh[j * rs + c] += scale * ds * k_bh[j * rs + c];"),
    ("bwd_g_from_keys", "dot += do_row[c] * v_bh[j * rs + c];", "dot += do_row[c] * k_bh[j * rs + c];"),
    ("bwd_weights_unnormalised", "for (int64_t j = 0; j < n; ++j) a[j] /= sum;", ""),
    ("bwd_score_scale_dropped", "a[j] = scale * dot;", "a[j] = dot;"),
]


@pytest.mark.parametrize("name,old,new", BWD_MUTANTS, ids=[m[0] for m in BWD_MUTANTS])
def test_bwd_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / f"{name}.c"
    mutated.write_text(src.replace(old, new), encoding="utf-8")
    mutant = oracle.Oracle(oracle.compile_source(str(mutated), str(tmp_path / f"lib{name}.so")))
    failed = []
    for check in oracle_bwd_pins.ALL_BWD_CHECKS:
        try:
            check(oracle.mha, mutant.mha_bwd)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every gradient pin"

