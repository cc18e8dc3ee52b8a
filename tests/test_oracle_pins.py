"""The fp64 oracle against its pins (closed forms, invariants, special cases, brute force).
CPU only."""
import pytest

import oracle.attnres_oracle as O
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(O)
