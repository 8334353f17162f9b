"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import pins
from oracle import dsa_oracle


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(dsa_oracle)
