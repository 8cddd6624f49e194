"""The fp64 oracle against hand-worked values, exact special cases,
invariants and library routines (see ``pins.py``).  CPU only."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)
