"""Pins of the CPU oracle against closed forms, brute force, library routines
and hand-derived values (no GPU needed)."""

import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, orc):
    pin(orc)
