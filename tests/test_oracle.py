"""The fp64 oracle against facts fixed by the mathematics (no GPU needed)."""
import pytest

import _pins


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()
