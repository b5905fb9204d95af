"""The transposed-convolution oracle against its pins (CPU only), and builds
with a planted mistake the pins must catch: 11 the stride's divisibility
not checked, 12 the kernel read flipped."""
import pytest

import oracle
from transpose_pins import TRANSPOSE_PINS


@pytest.mark.parametrize("pin", TRANSPOSE_PINS, ids=lambda p: p.__name__)
def test_transpose_pin(pin):
    pin(oracle.Oracle())


@pytest.mark.parametrize("mutant", [11, 12])
def test_transpose_mutant_is_caught(mutant):
    o = oracle.Oracle(mutant)
    failed = []
    for pin in TRANSPOSE_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every transposed-convolution pin"
