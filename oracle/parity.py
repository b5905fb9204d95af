"""The parity bar between a computed convolution and the oracle -- TEST
INFRASTRUCTURE ONLY.

The bar ("Convolution, pooling and resize", Tolerances table: conv 1e-5 in
float32, 2e-3 for half in and out with float32 accumulation, as a scaled
error) is read as |err| <= tol * sum |w x| per output, where the sum is the
oracle's ``scale``.  That bounds the error of the accumulated sum.  Three
further terms are allowed for steps after the sum, each derived from the
arithmetic rather than tuned:

* the activation multiplies an error in its argument by at most its
  Lipschitz constant L (1 for identity / relu / clip / sigmoid / tanh, the
  slope magnitudes for leaky-relu and hard-sigmoid, 1.1 for silu, 1.5 for
  hard-swish whose slope t/3 + 1/2 peaks at t = 3);
* the float32 epilogue rounds after each add and in the activation (whose
  exp / tanh may differ by a few ulp between libraries): 4 float32 ulps of
  |acc| + |bias| + |residual|, times L;
* the output is rounded to its element type on both sides, and two values
  that straddle a rounding boundary land one output ulp apart.
"""
from __future__ import annotations

import numpy as np

from . import to_float64, ulp

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def lipschitz(act: str, alpha: float = 0.0, beta: float = 0.0) -> float:
    if act == "silu":
        return 1.1
    if act == "hard_swish":
        return 1.5
    if act in ("leaky_relu", "hard_sigmoid"):
        return max(1.0, abs(alpha))
    return 1.0


def bound(ref: dict, dtype: str, act: str, alpha=0.0, beta=0.0, bias_abs=None, res_abs=None):
    """Per-output allowed |y - y_ref| for oracle result ``ref``."""
    L = lipschitz(act, alpha, beta)
    mag = np.abs(ref["acc"])
    if bias_abs is not None:
        mag = mag + bias_abs
    if res_abs is not None:
        mag = mag + res_abs
    y_ref = to_float64(ref["y"], dtype)
    return (L * TOL[dtype] * ref["scale"] + 4.0 * L * ulp(mag, "f32")
            + ulp(y_ref, dtype))


def _max_not_nan(a) -> float:
    a = np.asarray(a, dtype=np.float64)
    a = a[~np.isnan(a)]
    return float(a.max()) if a.size else 0.0


def compare(y, ref: dict, dtype: str, act: str, alpha=0.0, beta=0.0, bias=None,
            residual=None, co_index=None) -> dict:
    """Check ``y`` (numpy, same layout as ``ref['y']``: float32 or uint16 bits)
    against oracle result ``ref``.  ``bias`` / ``residual`` are the operands
    (numpy, element type) used to size the epilogue rounding term; for sampled
    outputs pass ``co_index`` (the output channel of each sample) and the
    residual values already gathered at the samples.

    Returns dict(ok, worst, max_scaled_err, n_bad, first_bad)."""
    yv = to_float64(np.asarray(y), dtype)
    rv = to_float64(ref["y"], dtype)
    if yv.shape != rv.shape:
        return {"ok": False, "reason": f"shape {yv.shape} != {rv.shape}"}
    bias_abs = None
    if bias is not None:
        b = np.abs(to_float64(bias, dtype))
        if co_index is not None:
            bias_abs = b[co_index]
        else:
            bias_abs = b.reshape(1, -1, 1, 1)
    res_abs = np.abs(to_float64(residual, dtype)) if residual is not None else None
    lim = bound(ref, dtype, act, alpha, beta, bias_abs, res_abs)
    err = np.abs(yv - rv)
    same_nonfinite = (~np.isfinite(yv)) & (yv == rv)
    bad = ~((err <= lim) | same_nonfinite)
    scale = ref["scale"]
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(scale > 0, err / np.where(scale > 0, scale, 1.0), 0.0)
    out = {
        "ok": not bool(bad.any()),
        "n_bad": int(bad.sum()),
        "max_scaled_err": _max_not_nan(scaled),
        "worst": _max_not_nan(err / lim),
    }
    if bad.any():
        i = np.unravel_index(int(np.argmax(bad)), bad.shape)
        out["first_bad"] = {"index": [int(v) for v in i], "got": float(yv[i]),
                            "want": float(rv[i]), "limit": float(lim[i]),
                            "scale": float(scale[i])}
    return out
