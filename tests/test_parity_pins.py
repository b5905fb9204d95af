"""The parity checker against its pins (CPU only), and planted mistakes in
copies of the checker that the pins must catch."""
import importlib.util
import os
import sys
import types

import numpy as np
import pytest

import oracle.parity as real_parity
from parity_pins import PARITY_PINS

_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "parity.py")


@pytest.mark.parametrize("pin", PARITY_PINS, ids=lambda p: p.__name__)
def test_parity_pin(pin):
    pin(real_parity)


def _mutant(old: str, new: str) -> types.ModuleType:
    """A copy of oracle/parity.py with one substitution, loaded as a module of
    the oracle package (so its relative imports resolve)."""
    src = open(_SRC).read()
    assert src.count(old) == 1, f"mutation site not found once: {old!r}"
    mod = types.ModuleType("oracle._parity_mutant")
    mod.__package__ = "oracle"
    mod.__file__ = _SRC
    exec(compile(src.replace(old, new), _SRC, "exec"), mod.__dict__)
    return mod


MUTANTS = {
    "scale_is_abs_acc": ('L * TOL[dtype] * ref["scale"]', 'L * TOL[dtype] * np.abs(ref["acc"])'),
    "lipschitz_twice": ('L * TOL[dtype] * ref["scale"]', 'L * L * TOL[dtype] * ref["scale"]'),
    "ulp_one_exponent_off": ("from . import to_float64, ulp",
                             "from . import to_float64\nfrom . import ulp as _u\n"
                             "def ulp(y, d):\n    return _u(y, d) * 2.0\n"),
    "bias_on_last_axis": ("bias_abs = b.reshape(1, -1, 1, 1)", "bias_abs = b.reshape(1, 1, 1, -1)"),
    "bias_ignores_co_index": ("bias_abs = b[co_index]", "bias_abs = b.max()"),
    "inf_passes_finite": ("same_nonfinite = (~np.isfinite(yv)) & (yv == rv)",
                          "same_nonfinite = ~np.isfinite(yv)"),
    "half_tol_loosened": ('"f16": 2e-3', '"f16": 2e-2'),
    "bf16_tol_loosened": ('"bf16": 2e-3', '"bf16": 4e-3'),
    "no_epilogue_term": ("+ 4.0 * L * ulp(mag, \"f32\")", "+ 0.0 * ulp(mag, \"f32\")"),
    "two_output_ulps": ("+ ulp(y_ref, dtype))", "+ 2.0 * ulp(y_ref, dtype))"),
    "residual_ignored": ("if res_abs is not None:\n        mag = mag + res_abs",
                         "if False:\n        mag = mag + res_abs"),
    "silu_slope_one": ('if act == "silu":\n        return 1.1', 'if act == "silu":\n        return 1.0'),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_parity_mutant_is_caught(name):
    mod = _mutant(*MUTANTS[name])
    failed = []
    for pin in PARITY_PINS:
        try:
            with np.errstate(invalid="ignore"):
                pin(mod)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"checker mutant {name} passed every pin"
