"""The oracle against its pins (CPU only): worked examples, closed forms,
invariants, torch float64 library routines and finite differences."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.get())
