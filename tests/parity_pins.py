"""Pins of the parity checker (``oracle.parity`` and ``oracle.ulp``): what
the bar accepts and rejects, checked against facts fixed outside the checker.

The bar for one output is

    |y - y_ref| <= L*tol*S + 4*L*ulp32(|acc| + |bias| + |residual|) + ulp_T(y_ref)

with tol = 1e-5 (float32) and 2e-3 (half, bfloat16 outputs) from the
"Convolution, pooling and resize" tolerance table, S = sum |w x|, L the
activation's Lipschitz constant, and ulp_T one unit in the last place of the
output type.  Each pin builds synthetic oracle results in which all terms but
one vanish, and asserts that an error of 0.99x that term passes and 1.01x fails
(or, for the output-ulp term, that one representable step passes and two do
not).  The expected sizes come from IEEE 754 / bfloat16 facts written out
here as constants (2^-23, 2^-10, 2^-7, the subnormal spacings), not from the
checker.

Each pin takes the checker module as its argument, so the same pins run
against the real checker and against copies with a planted mistake.
"""
from __future__ import annotations

import numpy as np
import torch

# One unit in the last place at 1.0, and the spacing of the subnormals
# (IEEE 754 binary32 / binary16, and bfloat16 = binary32's exponent with a
# 7-bit fraction).
ULP_AT_ONE = {"f32": 2.0 ** -23, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}
SUBNORMAL_STEP = {"f32": 2.0 ** -149, "f16": 2.0 ** -24, "bf16": 2.0 ** -133}
PAGE_TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}   # the tolerance table


def encode(values, dtype):
    """float64 values -> the operand array the checker reads (float32 values
    or uint16 bit patterns), rounded to nearest by numpy / torch."""
    v = np.asarray(values, dtype=np.float64)
    if dtype == "f32":
        return v.astype(np.float32)
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def decode(bits, dtype):
    if dtype == "f32":
        return np.asarray(bits, np.float64)
    if dtype == "f16":
        return np.asarray(bits).view(np.float16).astype(np.float64)
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ref_of(y_ref, acc, scale, dtype):
    shape = np.shape(y_ref)
    return {"y": encode(y_ref, dtype), "acc": np.broadcast_to(np.float64(acc), shape).copy(),
            "scale": np.broadcast_to(np.float64(scale), shape).copy(),
            "t": np.zeros(shape, np.float32)}


def verdicts(parity, y, ref, dtype, act="identity", alpha=0.0, **kw):
    """Per-element pass / fail of the checker (one output at a time)."""
    out = []
    for i in range(len(y)):
        r = {k: v[i:i + 1] for k, v in ref.items()}
        extra = {}
        for k, v in kw.items():
            extra[k] = v[i:i + 1] if (k in ("residual", "co_index") and v is not None) else v
        out.append(parity.compare(np.asarray(y)[i:i + 1], r, dtype, act, alpha, **extra)["ok"])
    return out


def representable_near(target, dtype):
    """The representable value of the type nearest to ``target`` (float64)."""
    return float(decode(encode([target], dtype), dtype)[0])


# ---------------------------------------------------------------------------
def pin_ulp_values(parity):
    """ulp at 1.0 and just below 2.0 is 2^-23 / 2^-10 / 2^-7; at 2.0 twice
    that; at 0 and deep in the subnormal range the subnormal spacing."""
    for dt in ("f32", "f16", "bf16"):
        u = parity.ulp(np.array([1.0, 1.5, 1.999, 2.0, -1.0]), dt)
        one = ULP_AT_ONE[dt]
        assert np.array_equal(u, [one, one, one, 2 * one, one]), (dt, u)
        sub = parity.ulp(np.array([0.0, SUBNORMAL_STEP[dt], 3 * SUBNORMAL_STEP[dt]]), dt)
        assert np.array_equal(sub, [SUBNORMAL_STEP[dt]] * 3), (dt, sub)
    # the largest half: 65504 = (2 - 2^-10) * 2^15, spacing 2^5
    assert parity.ulp(np.array([65504.0]), "f16")[0] == 32.0
    # the spacing is the gap to the next representable value
    for dt in ("f32", "f16", "bf16"):
        for v in (0.7, 3.0, 1000.0, 1e-3):
            step = float(parity.ulp(np.array([v]), dt)[0])
            lo = representable_near(v, dt)
            nxt = representable_near(lo + step, dt)
            assert nxt == lo + step, (dt, v, lo, step)


def pin_tolerance_term(parity):
    """With acc = 0 and y_ref = 0, the bar is tol*S (the page's tolerance) up to
    the subnormal spacing: 0.99x passes, 1.01x fails, in every element type."""
    for dt in ("f32", "f16", "bf16"):
        s = 512.0
        lim = PAGE_TOL[dt] * s
        ys = [representable_near(0.99 * lim, dt), representable_near(1.01 * lim, dt),
              -representable_near(0.99 * lim, dt), -representable_near(1.01 * lim, dt)]
        assert abs(ys[0]) < lim < abs(ys[1])
        ref = ref_of([0.0] * 4, 0.0, s, dt)
        assert verdicts(parity, encode(ys, dt), ref, dt) == [True, False, True, False], dt


def pin_lipschitz_once(parity):
    """The activation's Lipschitz constant multiplies the tolerance term once:
    silu 1.1, hard-swish 1.5, leaky-relu with alpha 3 gives 3."""
    dt = "f32"
    s = 1000.0
    for act, alpha, L in (("silu", 0.0, 1.1), ("hard_swish", 0.0, 1.5), ("leaky_relu", 3.0, 3.0),
                          ("relu", 0.0, 1.0), ("tanh", 0.0, 1.0)):
        lim = L * PAGE_TOL[dt] * s
        ys = [0.99 * lim, 1.01 * lim]
        ref = ref_of([0.0, 0.0], 0.0, s, dt)
        assert verdicts(parity, encode(ys, dt), ref, dt, act, alpha) == [True, False], act


def pin_epilogue_term(parity):
    """With S = 0 and y_ref = 0 the bar is 4*L*ulp32(|acc|+|bias|+|residual|):
    2^10 from the sum, the bias or the residual alone gives 4*2^-13."""
    for dt in ("f32", "f16"):
        lim = 4 * 2.0 ** -13
        ys = [representable_near(0.99 * lim, dt), representable_near(1.01 * lim, dt)]
        assert ys[0] < lim < ys[1]
        y = encode(ys, dt)
        # the magnitude from the sum
        assert verdicts(parity, y, ref_of([0.0, 0.0], 1024.0, 0.0, dt), dt) == [True, False]
        # ... from the bias of the output's channel (full layout: one channel)
        ref = ref_of(np.zeros((1, 2, 1, 1)), 0.0, 0.0, dt)
        ref["y"] = encode(np.zeros((1, 2, 1, 1)), dt)
        bias = encode([1024.0, 1024.0], dt)
        yy = encode(np.array(ys).reshape(1, 2, 1, 1), dt)
        got = parity.compare(yy, ref, dt, "identity", bias=bias)
        assert got["n_bad"] == 1 and got["first_bad"]["index"] == [0, 1, 0, 0], got
        # ... from the residual at that output
        res = encode(np.full((1, 2, 1, 1), -1024.0), dt)
        got = parity.compare(yy, ref, dt, "identity", residual=res)
        assert got["n_bad"] == 1 and got["first_bad"]["index"] == [0, 1, 0, 0], got
        # without bias or residual the same errors both fail
        got = parity.compare(yy, ref, dt, "identity")
        assert got["n_bad"] == 2, got


def pin_bias_channel_axis(parity):
    """The bias of output channel co sizes only that channel's outputs (NCHW:
    axis 1), in the full layout and, through co_index, for sampled outputs."""
    dt = "f32"
    lim = 4 * 2.0 ** -13
    bias = encode([0.0, 1024.0, 0.0], dt)       # only channel 1 has a large bias
    y = np.zeros((1, 3, 2, 2))
    y[0, :, 1, 0] = 0.99 * lim                  # one error per channel, 0.99x channel 1's limit
    ref = ref_of(np.zeros((1, 3, 2, 2)), 0.0, 0.0, dt)
    got = parity.compare(encode(y, dt), ref, dt, "identity", bias=bias)
    assert got["n_bad"] == 2 and got["first_bad"]["index"] == [0, 0, 1, 0], got
    # sampled: the same outputs as a flat list, each with its channel
    flat = np.arange(12)
    co = (flat // 4) % 3
    sref = {k: v.reshape(-1)[flat] for k, v in ref.items()}
    ok = verdicts(parity, encode(y, dt).reshape(-1)[flat], sref, dt, bias=bias, co_index=co)
    assert [i for i, v in enumerate(ok) if not v] == [2, 10], ok   # channels 0 and 2, row 1 col 0


def pin_output_ulp_term(parity):
    """Both sides round the result once to the output type: one representable
    step from y_ref passes, two fail (S = 0, acc = 0)."""
    for dt in ("f32", "f16", "bf16"):
        for yr in (1.0, -3.0, 0.3):
            base = representable_near(yr, dt)
            step = ULP_AT_ONE[dt] * 2.0 ** np.floor(np.log2(abs(base)))
            ys = [base + step, base + 2 * step, base - step]
            ref = ref_of([base] * 3, 0.0, 0.0, dt)
            got = verdicts(parity, encode(ys, dt), ref, dt)
            assert got == [True, False, True], (dt, yr, got)


def pin_nonfinite(parity):
    """An infinity passes only against the same infinity; NaN never passes;
    a finite value never passes against an infinite reference."""
    dt = "f32"
    ys = [np.inf, np.inf, -np.inf, np.nan, 1.0]
    refs = [np.inf, 1.0, np.inf, np.nan, np.inf]
    ref = ref_of(refs, 0.0, 1.0, dt)
    with np.errstate(invalid="ignore"):
        assert verdicts(parity, encode(ys, dt), ref, dt) == [True, False, False, False, False]


def pin_shape_mismatch(parity):
    """Outputs of another shape fail, whatever their values."""
    ref = ref_of(np.zeros((1, 2, 3, 3)), 0.0, 1.0, "f32")
    got = parity.compare(np.zeros((1, 2, 3, 4), np.float32), ref, "f32", "identity")
    assert not got["ok"]


def pin_scaled_error_report(parity):
    """max_scaled_err is max |err| / S over the outputs (the page's scaled
    error), independent of the other terms of the bar."""
    dt = "f32"
    ref = ref_of([0.0, 0.0, 0.0], 0.0, [100.0, 10.0, 1.0], dt)
    ref["scale"] = np.array([100.0, 10.0, 1.0])
    y = encode([1e-4, 5e-5, 2e-6], dt)
    got = parity.compare(y, ref, dt, "identity")
    assert abs(got["max_scaled_err"] - 5e-6) < 1e-12, got


PARITY_PINS = [pin_ulp_values, pin_tolerance_term, pin_lipschitz_once, pin_epilogue_term,
               pin_bias_channel_axis, pin_output_ulp_term, pin_nonfinite, pin_shape_mismatch,
               pin_scaled_error_report]
