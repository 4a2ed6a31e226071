"""The float64 oracle against what the pages and the mathematics fix.

Runs on CPU only.  Each pin is documented in ``tests/oracle_pins.py``.
"""

import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle)
