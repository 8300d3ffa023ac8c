"""The oracle's gradient against its pins (CPU only)."""
import pytest

import oracle
from tests import oracle_bwd_pins


@pytest.mark.parametrize("check", oracle_bwd_pins.ALL_BWD_CHECKS,
                         ids=[c.__name__ for c in oracle_bwd_pins.ALL_BWD_CHECKS])
def test_bwd_pin(check):
    check(oracle.mha, oracle.mha_bwd)
