"""Pins of the CPU oracle against closed forms, brute force, library routines
and hand-derived values (no GPU needed)."""

import pytest

import calib_pins
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, orc):
    pin(orc)


@pytest.mark.parametrize("pin", calib_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_calibration_pin(pin):
    from oracle import calibration
    pin(calibration)
