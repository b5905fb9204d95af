"""The pins catch plausible mistakes: each build of the oracle with one
planted mistake (see ORACLE_MUTANT in conv_oracle.c) fails at least one pin.

Mutants: 1 transposed kernel taps, 2 top pad used for the left border,
3 groups all read the first channel slice, 4 residual added before the bias,
5 dilation folded into the stride, 6 the +1 of the output size dropped,
7 the sum's sign flipped, 8 activation applied before the residual,
9 truncation instead of round-to-even, 10 clamp-to-edge border instead of
zeros.
"""
import pytest

import oracle
from oracle_pins import PINS

MUTANTS = list(range(1, 11))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_caught(mutant):
    o = oracle.Oracle(mutant)
    assert o.lib.oracle_mutant() == mutant
    failed = []
    for pin in PINS:
        try:
            pin(o)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"
