"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from oracle import arith
from oracle_pins import PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_mac_and_param_counts_exercise():
    """"Convolutions", section 7, exercise 1 and its printed solution, at 56x56."""
    # (a) 3x3 conv 64 -> 128: 73,856 params (with bias), ~231 M MACs
    assert arith.params(64, 128, 3, 3) == 73_856
    assert arith.macs(1, 64, 128, 3, 3, 56, 56) == 231_211_008
    # (b) depthwise 3x3: 576 params, ~1.8 M MACs; pointwise: 8,192 params, ~25.7 M MACs
    assert arith.params(64, 64, 3, 3, groups=64, bias=False) == 576
    assert round(arith.macs(1, 64, 64, 3, 3, 56, 56, groups=64) / 1e5) == 18
    assert arith.params(64, 128, 1, 1, bias=False) == 8_192
    assert round(arith.macs(1, 64, 128, 1, 1, 56, 56) / 1e5) == 257
    sep, std = arith.depthwise_separable_ratio(64, 128, 3, 56, 56)
    assert round(sep / std, 3) == 0.119
    assert sep * 1152 == std * 137          # exactly 1/128 + 1/9 (section 2.3)
    # (c) bottleneck 256 -> 64 -> 64 -> 256: ~69 K params, ~218 M MACs
    p = (arith.params(256, 64, 1, 1, bias=False) + arith.params(64, 64, 3, 3, bias=False)
         + arith.params(64, 256, 1, 1, bias=False))
    m = (arith.macs(1, 256, 64, 1, 1, 56, 56) + arith.macs(1, 64, 64, 3, 3, 56, 56)
         + arith.macs(1, 64, 256, 1, 1, 56, 56))
    assert round(p / 1000) == 70 and 68_000 < p < 70_000
    assert round(m / 1e6) == 218


def test_grouped_macs_divide_by_groups():
    """Section 2.3: grouped convolution costs 1/g of the dense one."""
    assert arith.macs(16, 512, 512, 3, 3, 28, 28, groups=32) * 32 == \
        arith.macs(16, 512, 512, 3, 3, 28, 28)


def test_oracle_thread_count_does_not_change_bits():
    o = oracle.Oracle()
    rng = np.random.default_rng(31)
    x = rng.uniform(-1, 1, (2, 6, 9, 9)).astype(np.float32)
    w = rng.uniform(-1, 1, (4, 3, 3, 3)).astype(np.float32)
    a = o.conv2d(x, w, pads=(1, 1, 1, 1), groups=2, nthreads=1)
    b = o.conv2d(x, w, pads=(1, 1, 1, 1), groups=2, nthreads=7)
    for k in a:
        assert np.array_equal(a[k], b[k])


def test_oracle_rejects_bad_geometry():
    o = oracle.Oracle()
    x = np.zeros((1, 3, 4, 4), np.float32)
    with pytest.raises(ValueError):
        o.conv2d(x, np.zeros((2, 2, 3, 3), np.float32))       # channels
    with pytest.raises(ValueError):
        o.conv2d(x, np.zeros((2, 3, 5, 5), np.float32))       # no output
