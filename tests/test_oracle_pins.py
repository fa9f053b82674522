"""The oracle against its pins (exact arithmetic, library routines, worked
examples and invariants): see ``pins.py``."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.lib())
