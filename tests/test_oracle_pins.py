"""The float64 oracle against what the pages and mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(oracle.mha)


def test_thread_count_changes_no_bit():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((3, 33, 4, 16))
    k = rng.standard_normal((3, 33, 4, 16))
    v = rng.standard_normal((3, 33, 4, 16))
    for mask in (0, 1, 2):
        lens = np.array([33, 5, 0], dtype=np.int32)
        o1 = oracle.mha(q, k, v, mask, key_lens=lens, threads=1)
        o8 = oracle.mha(q, k, v, mask, key_lens=lens, threads=8)
        assert np.array_equal(o1, o8)


def test_bad_arguments_rejected():
    q = np.zeros((1, 3, 1, 4))
    k = np.zeros((1, 5, 1, 4))
    with pytest.raises(ValueError):
        oracle.mha(q, k, k, mask_kind=1)          # causal needs Lq == Lk
    with pytest.raises(ValueError):
        oracle.mha(q, k, k, mask_kind=2)          # key padding needs key_lens
    with pytest.raises(ValueError):
        oracle.mha(q, k, k, mask_kind=5)          # unknown mask kind
