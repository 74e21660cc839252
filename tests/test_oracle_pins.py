"""The oracle against its pins (closed forms, invariants, brute force, planted keys)."""
import pytest

import oracle
from pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle.get())
