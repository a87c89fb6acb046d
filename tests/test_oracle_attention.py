"""The float64 attention oracle and the byte-move oracle against their pins."""

import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin_holds(pin):
    pin()
