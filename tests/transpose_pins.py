"""Pins of the transposed-convolution oracle: facts fixed outside its loop.

* output size ("Convolutions", sections 2.1 and 8: H_out = (H - 1)s - 2p + k,
  plus output_padding to pick which input size of a many-to-one forward map
  was meant -- 7 and 8 both map to 4 with k = 3, s = 2, p = 1);
* the checkerboard exercise of "Convolutions", section 8, exercise 3: an
  all-ones input and kernel with stride 2 give interior values 1, 2, 4 for
  k = 3 and a constant 4 for k = 4;
* the adjoint identity: <conv(x; w), y> = <x, conv_transpose(y; w)> for the
  same stride, pads, dilation and groups (the transposed convolution is the
  forward one's input-gradient, "Convolutions", section 2.4), against the
  pinned forward oracle;
* torch's conv_transpose2d on the CPU in float64 (section 3, How you'd test it).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def _rand(rng, shape):
    return rng.uniform(-1, 1, size=shape).astype(np.float32)


def pin_transpose_output_size(o):
    for h, k, p, s in ((4, 3, 1, 2), (7, 4, 1, 2), (10, 3, 0, 1), (5, 2, 0, 2), (28, 7, 3, 2)):
        assert o.transpose_extent(h, k, p, p, s, 1, 0) == (h - 1) * s - 2 * p + k
    assert o.transpose_extent(4, 3, 1, 1, 2, 1, 0) == 7
    assert o.transpose_extent(4, 3, 1, 1, 2, 1, 1) == 8
    # both are preimages of 4 under the forward map
    assert o.output_extent(7, 3, 1, 1, 2, 1) == 4 and o.output_extent(8, 3, 1, 1, 2, 1) == 4
    assert o.transpose_extent(5, 3, 0, 0, 1, 2, 0) == 9   # dilation: d(k - 1) + 1 = 5


def pin_transpose_checkerboard(o):
    ones = np.ones((1, 1, 6, 6), np.float32)
    y3 = o.conv_transpose2d(ones, np.ones((1, 1, 3, 3), np.float32), stride=(2, 2))["acc"][0, 0]
    inner = y3[2:-2, 2:-2]
    for i in range(inner.shape[0]):
        for j in range(inner.shape[1]):
            want = (2 if (i + 2) % 2 == 0 else 1) * (2 if (j + 2) % 2 == 0 else 1)
            assert inner[i, j] == want, (i, j, inner[i, j])
    assert set(np.unique(inner)) == {1.0, 2.0, 4.0}
    y4 = o.conv_transpose2d(ones, np.ones((1, 1, 4, 4), np.float32), stride=(2, 2))["acc"][0, 0]
    assert np.all(y4[2:-2, 2:-2] == 4.0)


def pin_transpose_adjoint(o):
    rng = np.random.default_rng(83)
    for (h, w, k, s, pads, d, g, cin, cout) in ((9, 8, 3, 2, (1, 1, 1, 1), (1, 1), 1, 3, 4),
                                                (11, 10, 4, (2, 3), (1, 2, 0, 1), (1, 2), 2, 4, 6),
                                                (7, 9, 3, (1, 1), (2, 0, 1, 2), (2, 1), 3, 6, 3),
                                                (8, 8, 1, (2, 2), (0, 0, 0, 0), (1, 1), 1, 5, 2)):
        st = s if isinstance(s, tuple) else (s, s)
        x = _rand(rng, (2, cin, h, w))
        wf = _rand(rng, (cout, cin // g, k, k))          # forward OIHW = transposed [C_in_T][C_out_T/g]
        fwd = o.conv2d(x, wf, stride=st, pads=pads, dilation=d, groups=g)["acc"]
        ho, wo = fwd.shape[2:]
        yv = _rand(rng, (2, cout, ho, wo))
        oph = (h + pads[0] + pads[2] - d[0] * (k - 1) - 1) % st[0]
        opw = (w + pads[1] + pads[3] - d[1] * (k - 1) - 1) % st[1]
        bwd = o.conv_transpose2d(yv, wf, stride=st, pads=pads, dilation=d, out_pad=(oph, opw), groups=g)["acc"]
        assert bwd.shape == x.shape, (bwd.shape, x.shape)
        lhs = float(np.sum(fwd * yv.astype(np.float64)))
        rhs = float(np.sum(x.astype(np.float64) * bwd))
        assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + 1.0), (lhs, rhs)


def pin_transpose_torch_float64(o):
    rng = np.random.default_rng(89)
    for (s, p, d, op, g, cin, cout, k) in ((2, 1, 1, 1, 1, 4, 6, 3), (2, 0, 1, 0, 2, 4, 6, 4),
                                           (3, 2, 2, 1, 3, 6, 9, 3), (1, 1, 1, 0, 1, 3, 5, 5),
                                           (2, 1, 1, 0, 4, 8, 8, 2)):
        x = _rand(rng, (2, cin, 7, 6))
        w = _rand(rng, (cin, cout // g, k, k))
        r = o.conv_transpose2d(x, w, stride=(s, s), pads=(p, p, p, p), dilation=(d, d), out_pad=(op, op), groups=g)
        ref = F.conv_transpose2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(), stride=s, padding=p,
                                 output_padding=op, groups=g, dilation=d).numpy()
        assert r["acc"].shape == ref.shape, (r["acc"].shape, ref.shape)
        assert np.all(np.abs(r["acc"] - ref) <= 1e-12 * (r["scale"] + 1e-300))


def pin_transpose_stride1_is_flipped_conv(o):
    """At stride 1 the transposed convolution is the forward one with the
    kernel flipped in both axes and channels swapped, padded by d(k-1) - p."""
    rng = np.random.default_rng(97)
    x = _rand(rng, (1, 3, 8, 7))
    w = _rand(rng, (3, 2, 3, 4))
    t = o.conv_transpose2d(x, w, pads=(1, 2, 0, 1))["acc"]
    wf = np.ascontiguousarray(np.flip(w, axis=(2, 3)).transpose(1, 0, 2, 3))
    f = o.conv2d(x, wf, pads=(2 - 1, 3 - 2, 2 - 0, 3 - 1))["acc"]
    assert t.shape == f.shape and np.allclose(t, f, rtol=0, atol=1e-12)


TRANSPOSE_PINS = [pin_transpose_output_size, pin_transpose_checkerboard, pin_transpose_adjoint,
                  pin_transpose_torch_float64, pin_transpose_stride1_is_flipped_conv]
