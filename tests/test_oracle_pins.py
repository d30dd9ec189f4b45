"""The CPU oracle against its pins (see ``oracle_pins.py``)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)
