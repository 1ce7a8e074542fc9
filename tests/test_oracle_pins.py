"""CPU pins of the float64 oracle (no GPU). Each test runs one pin from pins.py."""

import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=[p.__name__ for p in pins.ALL_PINS])
def test_pin(pin):
    pin()
