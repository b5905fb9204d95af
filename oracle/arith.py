"""Closed-form counts of a convolution layer -- TEST INFRASTRUCTURE ONLY.

"Convolutions", section 2.3 (parameters and FLOPs): a layer with Ci input and
Co output channels, a kh x kw kernel and g groups producing Ho x Wo outputs has
Co * (Ci/g) * kh * kw weights (+ Co biases) and Ho * Wo * Co * (Ci/g) * kh * kw
multiply-adds per image.  The depthwise-separable ratio of that section
follows from the same counts.  The benchmark's FLOP figure is twice the MAC
count over the whole batch.
"""
from __future__ import annotations


def macs(n, cin, cout, kh, kw, ho, wo, groups=1) -> int:
    return n * ho * wo * cout * (cin // groups) * kh * kw


def params(cin, cout, kh, kw, groups=1, bias=True) -> int:
    return cout * (cin // groups) * kh * kw + (cout if bias else 0)


def flops(n, cin, cout, kh, kw, ho, wo, groups=1) -> int:
    return 2 * macs(n, cin, cout, kh, kw, ho, wo, groups)


def depthwise_separable_ratio(cin, cout, k, ho, wo):
    """(MACs of a k x k depthwise + 1x1 pointwise pair, MACs of the dense k x k)."""
    sep = macs(1, cin, cin, k, k, ho, wo, groups=cin) + macs(1, cin, cout, 1, 1, ho, wo)
    std = macs(1, cin, cout, k, k, ho, wo)
    return sep, std
