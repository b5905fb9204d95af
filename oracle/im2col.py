"""Second, independent brute force of the convolution sum: unfold then multiply.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  This is a numpy
restatement of "Convolutions", section 2.4 (convolution as a matrix multiply:
cols = im2col(X) with one column of C*kh*kw taps per output position, then
Y = W cols per group) and the im2col description of its section 3 (a tap
index table over the zero-padded input, gathered in one step).  It is written
separately from the C nested loop so that the two can check each other:
padding here is a zero-padded copy, taps are gathered by index arrays, the
sum is a float64 matrix product.  Pads are per side (top, left, bottom,
right) and stride / dilation per axis.
"""
from __future__ import annotations

import numpy as np


def _extent(size, k, pad_begin, pad_end, stride, dil):
    return (size + pad_begin + pad_end - dil * (k - 1) - 1) // stride + 1


def unfold(x: np.ndarray, kh: int, kw: int, stride, pads, dilation) -> np.ndarray:
    """(B, C, H, W) float64 -> (B, C*kh*kw, Ho*Wo) columns, rows ordered (c, u, v)."""
    b, c, h, w = x.shape
    pt, pl, pb, pr = pads
    sh, sw = stride
    dh, dw = dilation
    ho = _extent(h, kh, pt, pb, sh, dh)
    wo = _extent(w, kw, pl, pr, sw, dw)
    xp = np.zeros((b, c, h + pt + pb, w + pl + pr), dtype=np.float64)
    xp[:, :, pt:pt + h, pl:pl + w] = x
    u, v = np.meshgrid(np.arange(kh), np.arange(kw), indexing="ij")
    i, j = np.meshgrid(np.arange(ho), np.arange(wo), indexing="ij")
    rows = i.reshape(1, -1) * sh + u.reshape(-1, 1) * dh   # (kh*kw, P)
    cols = j.reshape(1, -1) * sw + v.reshape(-1, 1) * dw   # (kh*kw, P)
    gathered = xp[:, :, rows, cols]                          # (B, C, kh*kw, P)
    return gathered.reshape(b, c * kh * kw, ho * wo), ho, wo


def conv2d_sum(x: np.ndarray, w: np.ndarray, stride=(1, 1), pads=(0, 0, 0, 0),
               dilation=(1, 1), groups=1) -> np.ndarray:
    """The raw convolution sum (no bias, residual or activation) in float64,
    one matrix product per group."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    b, cin, h, wd = x.shape
    cout, cin_g, kh, kw = w.shape
    assert cin_g * groups == cin and cout % groups == 0
    mg = cout // groups
    out = None
    for g in range(groups):
        cols, ho, wo = unfold(x[:, g * cin_g:(g + 1) * cin_g], kh, kw, stride, pads, dilation)
        wmat = w[g * mg:(g + 1) * mg].reshape(mg, -1)       # (Cout/g, Cin/g*kh*kw)
        if out is None:
            out = np.empty((b, cout, ho * wo), dtype=np.float64)
        out[:, g * mg:(g + 1) * mg] = np.einsum("ok,bkp->bop", wmat, cols)
    return out.reshape(b, cout, ho, wo)
