"""The ConvInteger oracle against its pins (CPU only), and builds of it with
one planted mistake each that the pins must catch: 21 padded taps as 0
instead of the zero point, 22 one weight zero point for every channel,
23 int8 read as uint8, 24 saturation instead of wrap-around, 25 x's zero
point ignored."""
import pytest

import oracle
from integer_pins import INTEGER_PINS


@pytest.mark.parametrize("pin", INTEGER_PINS, ids=lambda p: p.__name__)
def test_integer_pin(pin):
    pin(oracle.Oracle())


@pytest.mark.parametrize("mutant", [21, 22, 23, 24, 25])
def test_integer_mutant_is_caught(mutant):
    o = oracle.Oracle(mutant)
    assert o.lib.oracle_mutant() == mutant
    failed = []
    for pin in INTEGER_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every integer pin"
