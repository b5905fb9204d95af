"""Pins of the CPU oracle: checks against what the pages and the mathematics
fix, none of which re-derives the oracle's own formula.

Each pin is a function of an ``oracle.Oracle`` handle that raises
AssertionError when the handle disagrees with the fixed fact, so the same
pins run against the real oracle (test_oracle_pins.py) and against builds of
it with a planted mistake (test_oracle_mutants.py).
"""
from __future__ import annotations

import itertools
import os

import numpy as np
import torch
import torch.nn.functional as F

from oracle import im2col

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    mats, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] in ("input", "kernel", "output"):
                cur = parts[0]
                mats[cur] = []
                continue
            mats[cur].append([float(v) for v in parts])
    return {k: np.array(v) for k, v in mats.items()}


def _conv(o, x, w, **kw):
    """Raw sum through the oracle, float32 operands, identity epilogue."""
    return o.conv2d(np.asarray(x, np.float32), np.asarray(w, np.float32), **kw)


def _rand(rng, shape, lo=-1.0, hi=1.0):
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


# ---------------------------------------------------------------------------
def pin_output_size(o):
    """"Convolutions", section 2.1: the three printed checks (k=3 p=1 s=1 keeps
    H; 224 with k=7 p=3 s=2 gives 112; 10 with k=3 p=0 d=2 gives 6) and the
    worked example of section 1 (4 with k=3, no pad, stride 1 gives 2)."""
    for h in (1, 5, 56, 224):
        assert o.output_extent(h, 3, 1, 1, 1, 1) == h
    assert o.output_extent(224, 7, 3, 3, 2, 1) == 112
    assert o.output_extent(10, 3, 0, 0, 1, 2) == 6
    assert o.output_extent(4, 3, 0, 0, 1, 1) == 2
    # a window that does not fit yields no output
    assert o.output_extent(2, 3, 0, 0, 1, 1) == 0


def pin_worked_example(o):
    """"Convolutions", section 1: 4x4 input, 3x3 kernel -> 2x2, windows rows
    i..i+2 / cols j..j+2; hand-derived values in tests/golden."""
    for name in ("worked_example_4x4_3x3_ones.txt", "worked_example_4x4_3x3_ramp.txt"):
        g = _read_golden(name)
        r = _conv(o, g["input"][None, None], g["kernel"][None, None])
        assert r["y"].shape == (1, 1, 2, 2), r["y"].shape
        assert np.array_equal(r["acc"][0, 0], g["output"]), (name, r["acc"][0, 0])


def pin_im2col_brute_force(o):
    """"Convolutions", section 2.4: the sum equals W @ im2col(X) per group.  Tiny
    random shapes over every stride / pad / dilation / group combination up to
    3, asymmetric pads and kh != kw; agreement to 1e-12 of the scale."""
    rng = np.random.default_rng(7)
    cases = 0
    for (sh, sw), (dh, dw), groups in itertools.product(
            [(1, 1), (2, 1), (1, 3), (3, 2)], [(1, 1), (2, 1), (1, 3), (3, 2)], [1, 2, 3]):
        kh, kw = 1 + (sh + dh) % 3, 1 + (sw + 2 * dw) % 4
        pads = (sh % 3, dw % 3, (dh + 1) % 3, (sw + groups) % 3)
        cin, cout = 2 * groups, 3 * groups if groups > 1 else 4
        h, wd = 5 + groups, 7 - groups % 2
        if o.output_extent(h, kh, pads[0], pads[2], sh, dh) < 1:
            continue
        if o.output_extent(wd, kw, pads[1], pads[3], sw, dw) < 1:
            continue
        x = _rand(rng, (2, cin, h, wd))
        w = _rand(rng, (cout, cin // groups, kh, kw))
        r = _conv(o, x, w, stride=(sh, sw), pads=pads, dilation=(dh, dw), groups=groups)
        ref = im2col.conv2d_sum(x, w, (sh, sw), pads, (dh, dw), groups)
        assert r["acc"].shape == ref.shape, (r["acc"].shape, ref.shape)
        assert np.all(np.abs(r["acc"] - ref) <= 1e-12 * (r["scale"] + 1e-300)), \
            ((sh, sw), (dh, dw), groups)
        cases += 1
    assert cases >= 40


def pin_torch_cpu_float64(o):
    """Library cross-check: torch.nn.functional.conv2d on the CPU in float64
    ("Convolutions", section 3, How you'd test it: forward against F.conv2d for
    several stride / pad / dilation combinations and groups=6 depthwise)."""
    rng = np.random.default_rng(11)
    for stride, pad, dil, groups, cin, cout in [
            (1, 0, 1, 1, 3, 5), (2, 1, 1, 1, 4, 6), (1, 2, 2, 1, 2, 3),
            (2, 1, 2, 2, 4, 6), (1, 1, 1, 6, 6, 6), (1, 1, 1, 6, 6, 12), (3, 2, 1, 3, 6, 9)]:
        x = _rand(rng, (2, cin, 9, 8))
        w = _rand(rng, (cout, cin // groups, 3, 2))
        r = _conv(o, x, w, stride=(stride, stride), pads=(pad, pad, pad, pad),
                  dilation=(dil, dil), groups=groups)
        ref = F.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                       stride=stride, padding=pad, dilation=dil, groups=groups).numpy()
        assert r["acc"].shape == ref.shape
        assert np.all(np.abs(r["acc"] - ref) <= 1e-12 * (r["scale"] + 1e-300))
    # asymmetric pads: pad explicitly first, then an unpadded library conv
    x = _rand(rng, (1, 3, 7, 6))
    w = _rand(rng, (4, 3, 3, 3))
    pads = (2, 0, 1, 3)  # top, left, bottom, right
    r = _conv(o, x, w, pads=pads)
    xp = F.pad(torch.from_numpy(x).double(), (pads[1], pads[3], pads[0], pads[2]))
    ref = F.conv2d(xp, torch.from_numpy(w).double()).numpy()
    assert r["acc"].shape == ref.shape
    assert np.all(np.abs(r["acc"] - ref) <= 1e-12 * (r["scale"] + 1e-300))


def pin_all_ones_counts_taps(o):
    """With all-ones x and w every output is (Cin/g) x the number of its taps
    that land inside the image: a closed form per position that checks zero
    padding and the border of every axis independently ("Convolutions",
    section 2.1: taps at 0, d, ..., (k-1)d from each window start)."""
    for (h, wd, kh, kw, pads, (sh, sw), (dh, dw), g) in [
            (6, 5, 3, 3, (1, 1, 1, 1), (1, 1), (1, 1), 1),
            (7, 9, 5, 3, (2, 0, 3, 1), (2, 1), (1, 2), 2),
            (8, 8, 3, 3, (2, 2, 2, 2), (1, 1), (2, 2), 4),
            (5, 11, 1, 7, (0, 3, 0, 3), (1, 2), (1, 1), 1)]:
        cin, cout = 4, 4
        x = np.ones((1, cin, h, wd), np.float32)
        w = np.ones((cout, cin // g, kh, kw), np.float32)
        r = _conv(o, x, w, stride=(sh, sw), pads=pads, dilation=(dh, dw), groups=g)
        ho, wo = r["acc"].shape[2:]
        for i in range(ho):
            rows = sum(0 <= i * sh - pads[0] + u * dh < h for u in range(kh))
            for j in range(wo):
                cols = sum(0 <= j * sw - pads[1] + v * dw < wd for v in range(kw))
                assert np.all(r["acc"][0, :, i, j] == (cin // g) * rows * cols), (i, j)


def pin_delta_kernel_is_shift(o):
    """A kernel with a single 1 at tap (a, b) copies the input shifted by
    (a*d - pad_top, b*d - pad_left) and subsampled by the stride, zeros
    outside."""
    rng = np.random.default_rng(3)
    x = _rand(rng, (2, 1, 9, 10))
    for (kh, kw, a, b, pads, stride, dil) in [(3, 3, 0, 2, (1, 1, 1, 1), (1, 1), (1, 1)),
                                              (3, 4, 2, 1, (2, 0, 1, 2), (2, 1), (1, 2)),
                                              (5, 5, 4, 3, (0, 0, 0, 0), (1, 2), (1, 1))]:
        w = np.zeros((1, 1, kh, kw), np.float32)
        w[0, 0, a, b] = 1.0
        r = _conv(o, x, w, stride=stride, pads=pads, dilation=dil)
        ho, wo = r["acc"].shape[2:]
        for i in range(ho):
            for j in range(wo):
                ih = i * stride[0] - pads[0] + a * dil[0]
                iw = j * stride[1] - pads[1] + b * dil[1]
                want = x[:, 0, ih, iw] if (0 <= ih < 9 and 0 <= iw < 10) else 0.0
                assert np.all(r["acc"][:, 0, i, j] == want)


def pin_stride_subsamples(o):
    """A stride-s output is every s-th output of the stride-1 convolution with
    the same pads (window starts at 0, s, 2s, ...; section 2.1)."""
    rng = np.random.default_rng(5)
    x = _rand(rng, (1, 3, 11, 12))
    w = _rand(rng, (2, 3, 3, 2))
    pads = (1, 2, 1, 0)
    full = _conv(o, x, w, pads=pads)["acc"]
    for sh, sw in [(2, 2), (3, 1), (1, 3)]:
        r = _conv(o, x, w, pads=pads, stride=(sh, sw))["acc"]
        sub = full[:, :, ::sh, ::sw][:, :, :r.shape[2], :r.shape[3]]
        assert r.shape == sub.shape
        assert np.allclose(r, sub, rtol=0, atol=1e-12)


def pin_dilation_is_zero_inserted_kernel(o):
    """A rate-d kernel of size k equals a dense kernel of size d(k-1)+1 with
    zeros between the taps (section 2.1: taps at 0, d, ..., (k-1)d)."""
    rng = np.random.default_rng(9)
    x = _rand(rng, (1, 2, 12, 13))
    w = _rand(rng, (3, 2, 3, 2))
    for dh, dw in [(2, 2), (3, 1), (1, 2)]:
        dense = np.zeros((3, 2, dh * 2 + 1, dw * 1 + 1), np.float32)
        dense[:, :, ::dh, ::dw] = w
        a = _conv(o, x, w, dilation=(dh, dw), pads=(1, 1, 1, 1))["acc"]
        b = _conv(o, x, dense, pads=(1, 1, 1, 1))["acc"]
        assert a.shape == b.shape
        assert np.allclose(a, b, rtol=0, atol=1e-12)


def pin_groups_are_independent_slices(o):
    """Grouped convolution is g independent convolutions on channel slices;
    depthwise is g = C, and a channel multiplier m gives C*m outputs with
    output channel co reading input channel co // m ("Convolutions", sections
    2.3 and 3: one product per group)."""
    rng = np.random.default_rng(13)
    for g, cin, cout in [(2, 4, 6), (3, 6, 3), (5, 5, 5), (4, 4, 12)]:
        x = _rand(rng, (2, cin, 6, 7))
        w = _rand(rng, (cout, cin // g, 3, 3))
        r = _conv(o, x, w, pads=(1, 1, 1, 1), groups=g)["acc"]
        cg, mg = cin // g, cout // g
        for k in range(g):
            part = _conv(o, x[:, k * cg:(k + 1) * cg], w[k * mg:(k + 1) * mg],
                         pads=(1, 1, 1, 1))["acc"]
            assert np.array_equal(r[:, k * mg:(k + 1) * mg], part)


def pin_pointwise_is_matmul(o):
    """A 1x1, stride-1, unpadded convolution is the per-pixel matrix product
    W (Co x Ci) . X (Ci x HW) ("Convolutions", section 6: a 1x1 conv is
    already a GEMM)."""
    rng = np.random.default_rng(17)
    x = _rand(rng, (3, 5, 4, 6))
    w = _rand(rng, (7, 5, 1, 1))
    r = _conv(o, x, w)["acc"]
    ref = np.einsum("oc,bcp->bop", w[:, :, 0, 0].astype(np.float64),
                    x.reshape(3, 5, -1).astype(np.float64)).reshape(3, 7, 4, 6)
    assert np.allclose(r, ref, rtol=0, atol=1e-12)


def pin_scale_is_sum_of_abs_products(o):
    """The error scale is sum |w x|: equal to the sum itself for non-negative
    operands, and to the sum with |w|, |x| in general."""
    rng = np.random.default_rng(19)
    x = _rand(rng, (1, 3, 6, 6), 0.0, 1.0)
    w = _rand(rng, (2, 3, 3, 3), 0.0, 1.0)
    r = _conv(o, x, w, pads=(1, 1, 1, 1))
    assert np.allclose(r["scale"], r["acc"], rtol=1e-15, atol=0)
    xs = _rand(rng, (1, 3, 6, 6))
    ws = _rand(rng, (2, 3, 3, 3))
    a = _conv(o, xs, ws, pads=(1, 1, 1, 1))
    b = _conv(o, np.abs(xs), np.abs(ws), pads=(1, 1, 1, 1))
    assert np.allclose(a["scale"], b["acc"], rtol=1e-15, atol=0)


def pin_epilogue_order(o):
    """"Convolution, pooling and resize", Layout and operands: sum, bias,
    residual, activation, in that order, each step rounded to float32.
    Chosen values make every other order give a different float32 result."""
    one = np.ones((1, 1, 1, 1), np.float32)
    # acc = 1, bias = 2^24, residual = -2^24: float32 (1 + 2^24) rounds to 2^24,
    # so the ordered result is 0; adding the residual first would give 1.
    x = one.copy()
    w = one.copy()
    b = np.array([2.0 ** 24], np.float32)
    r = np.full((1, 1, 1, 1), -(2.0 ** 24), np.float32)
    res = o.conv2d(x, w, b, r)
    assert res["y"][0, 0, 0, 0] == 0.0, res["y"]
    # relu after the residual: acc + b = -3, r = +5 -> relu(2) = 2 (relu before
    # the residual would give 5)
    x2 = np.full((1, 1, 1, 1), -1.0, np.float32)
    res = o.conv2d(x2, np.full((1, 1, 1, 1), 2.0, np.float32), np.array([-1.0], np.float32),
                   np.full((1, 1, 1, 1), 5.0, np.float32), act="relu")
    assert res["y"][0, 0, 0, 0] == 2.0, res["y"]
    # the activation sees the bias: relu(-0.5 + 1) = 0.5
    res = o.conv2d(np.full((1, 1, 1, 1), -0.5, np.float32), one, np.array([1.0], np.float32),
                   act="relu")
    assert res["y"][0, 0, 0, 0] == 0.5
    # the sum itself is rounded to float32 before the bias is added
    x3 = np.array([[[[1.0, 2.0 ** -30]]]], np.float32)
    w3 = np.ones((1, 1, 1, 2), np.float32)
    res = o.conv2d(x3, w3, np.array([-1.0], np.float32))
    assert res["acc"][0, 0, 0, 0] == 1.0 + 2.0 ** -30
    assert res["y"][0, 0, 0, 0] == 0.0


def pin_activations(o):
    """ONNX activation definitions at points with exact float32 answers, plus
    the transcendental ones against numpy's float64 to within 4 float32 ulps."""
    A = o.activation
    assert A("identity", -3.5) == -3.5
    assert A("relu", -2.0) == 0.0 and A("relu", 3.0) == 3.0
    assert A("leaky_relu", -2.0, 0.1) == np.float32(-0.2) and A("leaky_relu", 2.0, 0.1) == 2.0
    assert A("clip", -7.0, -1.0, 6.0) == -1.0 and A("clip", 7.0, -1.0, 6.0) == 6.0
    assert A("clip", 2.5, -1.0, 6.0) == 2.5
    assert A("hard_swish", 3.0) == 3.0 and A("hard_swish", -3.0) == 0.0
    assert A("hard_swish", 4.0) == 4.0 and A("hard_swish", -4.0) == 0.0
    assert A("hard_swish", 0.0) == 0.0
    assert abs(A("hard_swish", 1.0) - 2.0 / 3.0) < 1e-7
    assert A("hard_sigmoid", 0.0, 0.2, 0.5) == 0.5
    assert A("hard_sigmoid", 10.0, 0.2, 0.5) == 1.0 and A("hard_sigmoid", -10.0, 0.2, 0.5) == 0.0
    assert A("hard_sigmoid", 1.0, 0.25, 0.5) == 0.75
    assert A("sigmoid", 0.0) == 0.5 and A("tanh", 0.0) == 0.0 and A("silu", 0.0) == 0.0
    ts = np.linspace(-12, 12, 97, dtype=np.float32)
    for t in ts:
        t64 = float(t)
        sig = 1.0 / (1.0 + np.exp(-t64))
        for name, want in (("sigmoid", sig), ("tanh", np.tanh(t64)), ("silu", t64 * sig)):
            got = A(name, float(t))
            assert abs(got - want) <= 4 * np.spacing(np.float32(abs(want))) + 1e-30, (name, t)


def pin_half_bf16_formats(o):
    """Exact decoding of every binary16 pattern against numpy's float16, and
    round-to-nearest-even encoding against numpy (half) and torch (bfloat16)
    on edge values and a random sweep."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([o.half_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert o.half_to_double(0x0001) == 2.0 ** -24 and o.half_to_double(0x7BFF) == 65504.0
    assert o.bf16_to_double(0x3F80) == 1.0 and o.bf16_to_double(0xC000) == -2.0
    edge = np.array([0.0, -0.0, 1.0, 65504.0, 65519.0, 65520.0, 1e9, 2.0 ** -24, 2.0 ** -25,
                     1.5 * 2.0 ** -25, 2.0 ** -26, 3.0 * 2.0 ** -25, 2.0 ** -14,
                     (1 + 2.0 ** -11), (1 + 3 * 2.0 ** -11), 6.1e-5, -2.5, 1e-8, np.inf, -np.inf],
                    dtype=np.float32)
    rng = np.random.default_rng(23)
    vals = np.concatenate([edge, (rng.standard_normal(20000) *
                                  np.exp2(rng.integers(-30, 18, 20000))).astype(np.float32)])
    with np.errstate(over="ignore"):
        want_h = vals.astype(np.float16).view(np.uint16)
    got_h = np.array([o.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got_h, want_h), vals[got_h != want_h][:5]
    want_b = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got_b = np.array([o.float_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got_b, want_b), vals[got_b != want_b][:5]


def pin_half_operands_decoded(o):
    """Half and bfloat16 operands are decoded exactly and the float32 result
    rounded once: a sum of exactly representable products gives the exact
    value in every element type."""
    x = np.array([[[[1.5, -0.25], [2.0, 0.125]]]], np.float32)
    w = np.array([[[[0.5, 2.0], [-1.0, 4.0]]]], np.float32)
    want = 1.5 * 0.5 - 0.25 * 2.0 - 2.0 + 0.125 * 4.0  # -1.25
    for dt, cast in (("f16", lambda a: a.astype(np.float16).view(np.uint16)),
                     ("bf16", lambda a: torch.from_numpy(a).to(torch.bfloat16)
                      .view(torch.int16).numpy().view(np.uint16))):
        r = o.conv2d(cast(x), cast(w), dtype=dt)
        assert r["acc"][0, 0, 0, 0] == want and r["t"][0, 0, 0, 0] == want
    # rounding of the output: 1 + 2^-11 is a half tie and rounds to even (1.0);
    # 1 + 3*2^-11 rounds up to 1 + 2^-9
    for v, want_bits in ((1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02)):
        r = o.conv2d(np.array([[[[1.0]]]], np.float16).view(np.uint16),
                     np.array([[[[1.0]]]], np.float16).view(np.uint16),
                     np.array([v - 1.0], np.float16).view(np.uint16), dtype="f16")
        # bias v-1 is exact in half (2^-11 and 3*2^-11 are representable)
        assert int(r["y"][0, 0, 0, 0]) == want_bits, hex(int(r["y"][0, 0, 0, 0]))


def pin_sampled_outputs_match_full(o):
    """Computing a chosen list of outputs gives the same bits as computing all
    of them (the sampled mode used on full-size workloads)."""
    rng = np.random.default_rng(29)
    x = _rand(rng, (2, 4, 7, 9))
    w = _rand(rng, (6, 2, 3, 3))
    b = _rand(rng, (6,))
    full = o.conv2d(x, w, b, pads=(1, 0, 2, 1), stride=(2, 1), groups=2, act="silu")
    idx = rng.choice(full["y"].size, 40, replace=False).astype(np.int64)
    part = o.conv2d(x, w, b, pads=(1, 0, 2, 1), stride=(2, 1), groups=2, act="silu", index=idx)
    for k in ("y", "acc", "scale", "t"):
        assert np.array_equal(part[k], full[k].reshape(-1)[idx])


PINS = [
    pin_output_size, pin_worked_example, pin_im2col_brute_force, pin_torch_cpu_float64,
    pin_all_ones_counts_taps, pin_delta_kernel_is_shift, pin_stride_subsamples,
    pin_dilation_is_zero_inserted_kernel, pin_groups_are_independent_slices,
    pin_pointwise_is_matmul, pin_scale_is_sum_of_abs_products, pin_epilogue_order,
    pin_activations, pin_half_bf16_formats, pin_half_operands_decoded,
    pin_sampled_outputs_match_full,
]
