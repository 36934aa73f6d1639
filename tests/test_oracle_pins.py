"""The CPU oracle against facts fixed outside it (format, library routine,
exact rationals, closed forms, invariants).  See oracle_pins.py."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle)
