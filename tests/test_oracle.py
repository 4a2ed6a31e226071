"""The float64 oracle against what the pages and the mathematics fix.

Runs on CPU only.  Each pin is documented in ``tests/oracle_pins.py``.
"""

import pytest

import oracle
import oracle.backward
import oracle.fp8
from oracle_pins import ALL_PINS, BWD_PINS, FP8_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle)


@pytest.mark.parametrize("pin", FP8_PINS, ids=[p.__name__ for p in FP8_PINS])
def test_fp8_pin(pin):
    pin(oracle.fp8)


@pytest.mark.parametrize("pin", BWD_PINS, ids=[p.__name__ for p in BWD_PINS])
def test_bwd_pin(pin):
    pin(oracle.backward, oracle)
