"""Second, independent brute force of the convolution sum: unfold then multiply.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  "Convolutions",
section 2.4, writes the convolution as one matrix product per group:
``Y_g = W_g . cols_g``, where ``W_g`` is the group's weights flattened to
(Cout/G) x (Cin/G * kh * kw) and ``cols_g`` has one column per output position
and one row per tap (channel c, kernel row u, kernel column v).  This module
builds that column matrix from its definition, one element at a time,

    cols[(c*kh + u)*kw + v, oh*Wo + ow] = x[c, oh*sh - pt + u*dh, ow*sw - pl + v*dw]
                                          (0 where that position is outside x),

and then multiplies in float64 with a library matrix product.  It shares
nothing with the C nested loop: here the taps become a matrix and the sum
is numpy's; there the sum runs over (c, u, v) in a fixed order.  Pads are per
side (top, left, bottom, right), stride and dilation per axis.
"""
from __future__ import annotations

import numpy as np


def output_extent(size: int, k: int, pad_begin: int, pad_end: int, stride: int, dil: int) -> int:
    """Window starts 0, s, 2s, ... of a padded axis whose span d(k-1)+1 still
    fits ("Convolutions", section 2.1)."""
    span = dil * (k - 1) + 1
    padded = size + pad_begin + pad_end
    count = 0
    start = 0
    while start + span <= padded:
        count += 1
        start += stride
    return count


def column_matrix(x: np.ndarray, kh: int, kw: int, stride, pads, dilation):
    """One image's channels (C, H, W) -> the (C*kh*kw, Ho*Wo) column matrix."""
    c_n, h, w = x.shape
    pt, pl, pb, pr = pads
    sh, sw = stride
    dh, dw = dilation
    ho = output_extent(h, kh, pt, pb, sh, dh)
    wo = output_extent(w, kw, pl, pr, sw, dw)
    cols = np.zeros((c_n * kh * kw, ho * wo), dtype=np.float64)
    for c in range(c_n):
        for u in range(kh):
            for v in range(kw):
                row = (c * kh + u) * kw + v
                for oh in range(ho):
                    ih = oh * sh - pt + u * dh
                    if ih < 0 or ih >= h:
                        continue  # the whole output row reads padding for this tap
                    for ow in range(wo):
                        iw = ow * sw - pl + v * dw
                        if 0 <= iw < w:
                            cols[row, oh * wo + ow] = x[c, ih, iw]
    return cols, ho, wo


def conv2d_sum(x: np.ndarray, w: np.ndarray, stride=(1, 1), pads=(0, 0, 0, 0),
               dilation=(1, 1), groups=1) -> np.ndarray:
    """The raw convolution sum (no bias, residual or activation) in float64:
    for every image and group, the weight matrix times the column matrix."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    b, cin, h, wd = x.shape
    cout, cin_g, kh, kw = w.shape
    assert cin_g * groups == cin and cout % groups == 0
    mg = cout // groups
    ho = output_extent(h, kh, pads[0], pads[2], stride[0], dilation[0])
    wo = output_extent(wd, kw, pads[1], pads[3], stride[1], dilation[1])
    out = np.zeros((b, cout, ho * wo), dtype=np.float64)
    for img in range(b):
        for g in range(groups):
            cols, _, _ = column_matrix(x[img, g * cin_g:(g + 1) * cin_g], kh, kw, stride, pads,
                                       dilation)
            wmat = w[g * mg:(g + 1) * mg].reshape(mg, cin_g * kh * kw)
            out[img, g * mg:(g + 1) * mg] = wmat @ cols
    return out.reshape(b, cout, ho, wo)
