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


def auto_pad(size: int, k: int, stride: int, dilation: int, mode: str) -> tuple[int, int]:
    """ONNX Conv auto_pad ("Convolution, pooling and resize", Layout and
    operands: auto_pad is turned into explicit pads), one axis.

    VALID: no padding.  SAME_UPPER / SAME_LOWER: pad so that the output has
    ceil(size / stride) positions; the total padding is what the last window
    needs beyond the input, split in two halves, the odd one at the end
    (SAME_UPPER) or at the beginning (SAME_LOWER).  Returns (begin, end)."""
    if mode == "VALID":
        return 0, 0
    out = -(-size // stride)
    span = dilation * (k - 1) + 1
    total = max(0, (out - 1) * stride + span - size)
    small, large = total // 2, total - total // 2
    if mode == "SAME_UPPER":
        return small, large
    if mode == "SAME_LOWER":
        return large, small
    raise ValueError(mode)
