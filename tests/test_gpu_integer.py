"""ConvInteger on the GPU against the CPU oracle, bit for bit ("Convolution,
pooling and resize", ConvInteger: exact int32 with wrap-around, tested bit for
bit against a plain definition over shapes, dilation, asymmetric padding,
groups, extreme values and all four type combinations)."""
import ctypes
import dataclasses
import zlib

import numpy as np
import pytest
import torch

import implicit_gemm_cnn_gb300 as conv
from gpu_util import orc
from workloads import INT_LAYERS, make_int_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _np(t):
    return t.cpu().numpy()


def _run(inp, **g):
    dev = {k: v.cuda() for k, v in inp.items()}
    y = conv.conv_integer2d(dev["x"], dev["w"], dev["x_zero"], dev["w_zero"], **g)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _oracle(inp, index=None, stride=1, pads=0, dilation=1, groups=1):
    wz = _np(inp["w_zero"]).astype(np.int64)
    return orc().conv_integer(_np(inp["x"]), _np(inp["w"]), int(_np(inp["x_zero"])[0]),
                              wz if wz.size > 1 else int(wz[0]), stride=conv._pair(stride),
                              pads=conv._pads(pads), dilation=conv._pair(dilation), groups=groups, index=index)


def _inputs(xs, ws, xt, wt, seed, per_channel=True, extreme=False):
    gen = torch.Generator().manual_seed(seed)
    rng = {"u8": (0, 256, torch.uint8), "i8": (-128, 128, torch.int8)}
    xl, xh, xd = rng[xt]
    wl, wh, wd = rng[wt]
    if extreme:  # only the ends of each range
        x = torch.where(torch.rand(xs, generator=gen) < 0.5, xl, xh - 1).to(xd)
        w = torch.where(torch.rand(ws, generator=gen) < 0.5, wl, wh - 1).to(wd)
    else:
        x = torch.randint(xl, xh, xs, generator=gen).to(xd)
        w = torch.randint(wl, wh, ws, generator=gen).to(wd)
    xz = torch.randint(xl, xh, (1,), generator=gen).to(xd)
    wz = torch.randint(wl, wh, (ws[0] if per_channel else 1,), generator=gen).to(wd)
    return {"x": x, "w": w, "x_zero": xz, "w_zero": wz}


CASES = [
    # (name, x shape, w shape, geometry)
    ("plain_3x3", (2, 16, 9, 11), (24, 16, 3, 3), dict(pads=1)),
    ("stride_dil_asym", (1, 8, 17, 19), (16, 8, 3, 3), dict(stride=(3, 2), pads=(1, 2, 0, 1), dilation=(2, 3))),
    ("grouped", (2, 12, 9, 10), (18, 4, 3, 3), dict(pads=1, groups=3)),
    ("depthwise", (2, 6, 11, 9), (12, 1, 5, 5), dict(pads=2, groups=6)),
    ("one_d", (3, 20, 1, 37), (30, 20, 1, 3), dict(stride=(1, 2), pads=(0, 1, 0, 1))),
    ("k_not_words", (1, 3, 13, 13), (200, 3, 7, 7), dict(stride=2, pads=3)),
    ("pointwise_tiles", (4, 64, 7, 9), (130, 64, 1, 1), dict()),
]


@pytest.mark.parametrize("types", [("u8", "u8"), ("u8", "i8"), ("i8", "u8"), ("i8", "i8")])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("per_channel", [False, True])
def test_conv_integer_bit_exact(case, types, per_channel):
    name, xs, ws, g = case
    inp = _inputs(xs, ws, *types, seed=zlib.crc32(name.encode()) % 997 + 7 * per_channel, per_channel=per_channel)
    assert np.array_equal(_run(inp, **g), _oracle(inp, **g))


@pytest.mark.parametrize("types", [("u8", "u8"), ("i8", "i8"), ("u8", "i8"), ("i8", "u8")])
def test_conv_integer_wraps_around(types):
    """Every term (x - x_zero)(w - w_zero) at +-255*255 over k = 4096*9: the
    interior sums pass 2^31 and wrap modulo 2^32, exactly as the definition's
    int32; border outputs (fewer taps) stay below."""
    hi = {"u8": (255, 0, torch.uint8), "i8": (127, -128, torch.int8)}
    xv, xz, xd = hi[types[0]]
    wv, wz, wd = hi[types[1]]
    inp = {"x": torch.full((1, 4096, 3, 4), xv, dtype=xd), "w": torch.full((2, 4096, 3, 3), wv, dtype=wd),
           "x_zero": torch.tensor([xz], dtype=xd), "w_zero": torch.tensor([wz, wz], dtype=wd)}
    y = _run(inp, pads=1)
    ref = _oracle(inp, pads=1)
    assert np.array_equal(y, ref)
    exact = 4096 * 9 * 255 * 255          # an interior output's sum
    assert int(ref[0, 0, 1, 1]) == ((exact + 2 ** 31) % 2 ** 32) - 2 ** 31 != exact


def test_conv_integer_workload_reduced_all_outputs():
    L = dataclasses.replace(INT_LAYERS["whisper_conv2_u8i8"], n=1, w=300)
    inp = make_int_inputs(L)
    g = dict(stride=L.stride, pads=L.pads, dilation=L.dilation, groups=L.groups)
    assert np.array_equal(_run(inp, **g), _oracle(inp, **g))


def test_conv_integer_workload_full_size_sampled():
    L = INT_LAYERS["whisper_conv2_u8i8"]
    inp = make_int_inputs(L)
    g = dict(stride=L.stride, pads=L.pads, dilation=L.dilation, groups=L.groups)
    y = _run(inp, **g)
    rng = np.random.default_rng(3)
    idx = np.unique(np.concatenate([rng.integers(0, y.size, 3000), [0, y.size - 1]])).astype(np.int64)
    assert np.array_equal(y.reshape(-1)[idx], _oracle(inp, index=idx, **g))
    y2 = _run(inp, **g)
    assert np.array_equal(y, y2)   # exact integers: the same bits every run


def test_conv_integer_rejects_float_epilogue_and_bad_zero_points():
    lib = conv.load()
    x = torch.zeros((1, 2, 5, 5), dtype=torch.uint8, device="cuda")
    w = torch.zeros((3, 2, 3, 3), dtype=torch.int8, device="cuda")
    z = torch.zeros((3,), dtype=torch.int8, device="cuda")
    y = torch.empty((1, 3, 3, 3), dtype=torch.int32, device="cuda")
    s = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    p = conv.make_problem(x.shape, w.shape, act="relu")
    st = lib.conv_integer_forward(ctypes.byref(p), 0, 1, x.data_ptr(), w.data_ptr(), x.data_ptr(), z.data_ptr(), 1,
                                  y.data_ptr(), s.data_ptr(), s.numel(), None)
    assert conv.STATUS[st] == "CONV_ERR_ARG"
    p = conv.make_problem(x.shape, w.shape)
    st = lib.conv_integer_forward(ctypes.byref(p), 0, 1, x.data_ptr(), w.data_ptr(), x.data_ptr(), z.data_ptr(), 2,
                                  y.data_ptr(), s.data_ptr(), s.numel(), None)
    assert conv.STATUS[st] == "CONV_ERR_ARG"        # two zero points for three channels
    st = lib.conv_integer_forward(ctypes.byref(p), 2, 1, x.data_ptr(), w.data_ptr(), x.data_ptr(), z.data_ptr(), 1,
                                  y.data_ptr(), s.data_ptr(), s.numel(), None)
    assert conv.STATUS[st] == "CONV_ERR_DTYPE"
    st = lib.conv_integer_forward(ctypes.byref(p), 0, 1, x.data_ptr(), w.data_ptr(), x.data_ptr(), z.data_ptr(), 1,
                                  y.data_ptr(), s.data_ptr(), 16, None)
    assert conv.STATUS[st] == "CONV_ERR_SCRATCH"
