"""Pins of the ConvInteger oracle: facts fixed outside its nested loop.

"Convolution, pooling and resize", ConvInteger: y = sum (x - xZero) *
(w - wZero[m]) in int32 with wrap-around, uint8 / int8 operands in any mix,
x's zero point one value, w's one value or one per output channel; a padded
tap is the real value zero (the quantized value xZero) and adds nothing.

Each pin is a function of an ``oracle.Oracle`` handle (the real oracle, or a
build with a planted mistake).
"""
from __future__ import annotations

import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    mats, cur = {}, None
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        if line in ("input", "kernel", "output"):
            cur = line
            mats[cur] = []
            continue
        mats[cur].append([int(v) for v in line.split()])
    return {k: np.array(v) for k, v in mats.items()}


def _wrap32(v: int) -> int:
    """An exact integer reduced modulo 2^32 to two's-complement int32."""
    v &= 0xFFFFFFFF
    return v - (1 << 32) if v >= (1 << 31) else v


def pin_integer_worked_example(o):
    """The 4x4 / 3x3 example with zero points 3 (x, uint8) and -1 (w, int8),
    worked by hand in tests/golden."""
    g = _golden("conv_integer_worked_example.txt")
    y = o.conv_integer(g["input"].astype(np.uint8)[None, None], g["kernel"].astype(np.int8)[None, None],
                       x_zero=3, w_zero=-1)
    assert np.array_equal(y[0, 0], g["output"]), y


def pin_integer_matches_float_definition(o):
    """Without overflow the int32 result is the exact integer sum: torch's
    float64 conv2d on the zero-point-subtracted operands (zero padding of
    x - xZero is padding x with xZero) over every type mix, strides,
    dilations, groups and per-channel zero points."""
    rng = np.random.default_rng(61)
    for xs, ws in ((False, False), (False, True), (True, False), (True, True)):
        for stride, pad, dil, groups in ((1, 1, 1, 1), (2, (1, 2), 1, 2), ((1, 2), 0, (2, 1), 3), (1, 2, 2, 6)):
            cin, cout = 6, 12 if groups != 6 else 6
            x = rng.integers(-128 if xs else 0, 128 if xs else 256, (2, cin, 9, 8)).astype(np.int8 if xs else np.uint8)
            w = rng.integers(-128 if ws else 0, 128 if ws else 256, (cout, cin // groups, 3, 2)).astype(
                np.int8 if ws else np.uint8)
            xz = int(rng.integers(-128 if xs else 0, 128 if xs else 256))
            wz = rng.integers(-128 if ws else 0, 128 if ws else 256, cout)
            st = stride if isinstance(stride, tuple) else (stride, stride)
            dl = dil if isinstance(dil, tuple) else (dil, dil)
            pd = pad if isinstance(pad, tuple) else (pad, pad)
            y = o.conv_integer(x, w, xz, wz, stride=st, pads=(pd[0], pd[1], pd[0], pd[1]), dilation=dl,
                               groups=groups)
            xt = torch.from_numpy(x.astype(np.float64) - xz)
            wt = torch.from_numpy(w.astype(np.float64) - wz.reshape(-1, 1, 1, 1))
            ref = F.conv2d(xt, wt, stride=st, padding=pd, dilation=dl, groups=groups).numpy()
            assert np.abs(ref).max() < 2 ** 31
            assert np.array_equal(y, ref.astype(np.int32)), (xs, ws, stride, pad, dil, groups)


def pin_integer_wraps_around(o):
    """A sum past 2^31 wraps modulo 2^32: 4096 channels x 3 x 3 taps of
    255 * 255 sum to 2,397,081,600, which an int32 holds as that minus 2^32."""
    x = np.full((1, 4096, 3, 3), 255, np.uint8)
    w = np.full((2, 4096, 3, 3), 255, np.uint8)
    y = o.conv_integer(x, w, 0, [0, 1])
    assert int(y[0, 0, 0, 0]) == _wrap32(4096 * 9 * 255 * 255) == 2_397_081_600 - 2 ** 32
    assert int(y[0, 1, 0, 0]) == _wrap32(4096 * 9 * 255 * 254)
    x2 = np.full((1, 4096, 3, 3), -128, np.int8)
    w2 = np.full((1, 4096, 3, 3), 127, np.int8)
    y2 = o.conv_integer(x2, w2, 127, -128)   # (-255) * 255 per term
    assert int(y2[0, 0, 0, 0]) == _wrap32(-4096 * 9 * 255 * 255)


def pin_integer_padding_is_the_zero_point(o):
    """x = xZero + 1 everywhere and w = wZero + 1: every in-bounds tap adds
    one, padded taps nothing -- the closed form (Cin/g) x in-bounds taps."""
    for (h, wd, k, pads, s, d, g) in ((6, 5, 3, (1, 1, 1, 1), (1, 1), (1, 1), 1),
                                      (7, 9, 5, (2, 0, 3, 1), (2, 1), (1, 2), 2)):
        x = np.full((1, 4, h, wd), 201, np.uint8)      # xZero = 200
        w = np.full((4, 4 // g, k, k), -6, np.int8)    # wZero = -7
        y = o.conv_integer(x, w, 200, -7, stride=s, pads=pads, dilation=d, groups=g)
        for i in range(y.shape[2]):
            rows = sum(0 <= i * s[0] - pads[0] + u * d[0] < h for u in range(k))
            for j in range(y.shape[3]):
                cols = sum(0 <= j * s[1] - pads[1] + v * d[1] < wd for v in range(k))
                assert np.all(y[0, :, i, j] == (4 // g) * rows * cols), (i, j)


def pin_integer_zero_points_cancel(o):
    """x equal to its zero point gives 0 whatever w; an output channel whose
    weights equal its own zero point gives 0; a per-channel zero point acts
    on its channel only."""
    rng = np.random.default_rng(67)
    w = rng.integers(-128, 128, (3, 2, 3, 3)).astype(np.int8)
    y = o.conv_integer(np.full((1, 2, 5, 5), 17, np.uint8), w, 17, [5, -3, 0], pads=(1, 1, 1, 1))
    assert not y.any()
    x = rng.integers(0, 256, (1, 2, 5, 5)).astype(np.uint8)
    w2 = w.copy()
    w2[1] = -3
    y2 = o.conv_integer(x, w2, 9, [5, -3, 0], pads=(1, 1, 1, 1))
    assert not y2[0, 1].any() and y2[0, 0].any() and y2[0, 2].any()


def pin_integer_int8_decoding(o):
    """int8 operands are two's complement: the byte 0xff is -1 (x) and 0x80
    is -128 (w): (-1 - 0) * (-128 - 0) = 128 per tap."""
    x = np.full((1, 1, 2, 2), -1, np.int8)
    w = np.full((1, 1, 2, 2), -128, np.int8)
    assert int(o.conv_integer(x, w, 0, 0)[0, 0, 0, 0]) == 4 * 128
    xu = x.view(np.uint8)   # the same bytes as uint8: 255
    assert int(o.conv_integer(xu, w, 0, 0)[0, 0, 0, 0]) == 4 * 255 * -128


def pin_integer_sampled_matches_full(o):
    """Computing a chosen list of outputs gives the bits of computing all."""
    rng = np.random.default_rng(71)
    x = rng.integers(0, 256, (2, 4, 7, 9)).astype(np.uint8)
    w = rng.integers(-128, 128, (6, 2, 3, 3)).astype(np.int8)
    wz = rng.integers(-128, 128, 6)
    full = o.conv_integer(x, w, 99, wz, pads=(1, 0, 2, 1), stride=(2, 1), groups=2)
    idx = rng.choice(full.size, 40, replace=False).astype(np.int64)
    part = o.conv_integer(x, w, 99, wz, pads=(1, 0, 2, 1), stride=(2, 1), groups=2, index=idx)
    assert np.array_equal(part, full.reshape(-1)[idx])


INTEGER_PINS = [pin_integer_worked_example, pin_integer_matches_float_definition, pin_integer_wraps_around,
                pin_integer_padding_is_the_zero_point, pin_integer_zero_points_cancel,
                pin_integer_int8_decoding, pin_integer_sampled_matches_full]
