"""The CPU oracle against the pages' worked examples, closed forms,
invariants, library routines and brute force (no GPU)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load_library())
