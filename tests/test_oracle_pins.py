"""The CPU oracle against its pins: golden cases, brute force, closed forms, invariants and
library routines for special cases. No GPU is involved."""

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.get())
