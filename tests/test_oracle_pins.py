"""The CPU oracle against the closed forms, invariants, library routines and
brute-force loops that the operator's definition fixes (no GPU)."""
import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle)
