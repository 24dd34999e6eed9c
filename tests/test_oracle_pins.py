"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import oracle.masw_oracle as o
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(o)
