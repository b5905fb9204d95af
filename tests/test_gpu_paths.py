"""Paths the C ABI promises beyond the aligned, unchained calls of the other
parity tests, each checked against the CPU oracle element by element.

* Operands at element offsets inside larger buffers ("Convolution, pooling and
  resize", Layout and operands: operands are buffers plus element offsets).
  Such pointers are legal and select other code: the gather tensor-core
  kernel instead of the shifted-window one, narrower (8- or 4-byte) or
  element copies in the depthwise kernel, the synchronous staging of the
  narrow depthwise kernel, the CUDA-core pointwise kernel without 16-byte B
  copies, scalar stores of the output.
* Chained layers: the ResNet-50 bottleneck pair (3x3 then 1x1 with residual)
  and the MobileNetV3 block (5x5 depthwise then 1x1), the second layer reading
  the first one's output on the GPU; its oracle reads that same tensor.
"""
import ctypes
import dataclasses
import zlib

import pytest
import torch

import implicit_gemm_cnn_gb300 as conv
from gpu_util import check_full, check_sampled
from workloads import LAYERS, make_inputs, random_layer_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _placed(t, off):
    """A device buffer holding t's elements from element `off` on, and the
    address of that element."""
    buf = torch.zeros(t.numel() + off + 16, dtype=t.dtype, device="cuda")
    buf[off:off + t.numel()].copy_(t.reshape(-1).to("cuda"))
    return buf, buf.data_ptr() + off * t.element_size()


def _run_offsets(inp, dtype, offs, flags=0, **g):
    """conv_forward with x / y / residual at element offsets offs = (ox, oy, orr)."""
    x, w, b, r = inp["x"], inp["w"], inp.get("bias"), inp.get("residual")
    p = conv.make_problem(x.shape, w.shape, dtype=dtype, has_bias=b is not None,
                          has_residual=r is not None, flags=flags, **g)
    ho, wo = conv.conv_output_shape(p)
    yshape = (x.shape[0], w.shape[0], ho, wo)
    ox, oy, orr = offs
    xbuf, xp = _placed(x, ox)
    ybuf, yp = _placed(torch.zeros(yshape, dtype=x.dtype), oy)
    rbuf, rp = _placed(r, orr) if r is not None else (None, None)
    wd = w.cuda()
    bd = b.cuda() if b is not None else None
    need = conv.conv_scratch_bytes(p)
    scratch = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    conv.conv_forward(p, xp, wd, bd, rp, yp, scratch if need else None, need)
    torch.cuda.synchronize()
    n = 1
    for v in yshape:
        n *= v
    return ybuf[oy:oy + n].view(yshape).cpu(), p


def _desc(p):
    return conv.conv_describe_variant(p)


# (name, x shape, w shape, geometry, dtypes, offsets (x, y, residual), residual?)
OFFSET_CASES = [
    # shifted-window layer shapes with x or y off 16 bytes: the gather kernel runs
    ("window_x_off", (2, 16, 12, 16), (40, 16, 3, 3), dict(pads=1, act="silu"), ("f16", "bf16"), (1, 0, 0), True),
    ("window_y_off", (2, 16, 12, 16), (40, 16, 3, 3), dict(pads=1, act="silu"), ("f16", "bf16"), (0, 1, 1), True),
    ("window_stem_x_off", (2, 3, 40, 48), (16, 3, 7, 7), dict(stride=2, pads=3, act="relu"), ("f16",), (3, 5, 0),
     False),
    # the pointwise tensor-core kernel: residual, x (element staging) and y (single stores) off 4 bytes
    ("pw_1x1_res_off", (2, 32, 8, 16), (64, 32, 1, 1), dict(act="relu"), ("bf16",), (0, 0, 1), True),
    ("pw_1x1_x_off", (2, 40, 9, 12), (48, 40, 1, 1), dict(act="silu"), ("f16",), (1, 0, 0), False),
    ("pw_1x1_y_off", (2, 24, 8, 10), (56, 24, 1, 1), dict(), ("f16", "bf16"), (0, 1, 0), True),
    # general depthwise kernel: 16-, 8-, 4-byte and element copies of x rows
    ("dw_general_f32_off2", (2, 6, 12, 10), (18, 1, 3, 3), dict(stride=(2, 1), pads=1, groups=6, act="relu"),
     ("f32",), (2, 1, 0), False),
    ("dw_general_f32_off1", (2, 6, 12, 10), (18, 1, 3, 3), dict(stride=(2, 1), pads=1, groups=6, act="relu"),
     ("f32",), (1, 3, 0), False),
    ("dw_general_half_off1", (2, 6, 12, 10), (18, 1, 3, 3), dict(stride=(2, 1), pads=1, groups=6),
     ("f16", "bf16"), (1, 1, 0), False),
    ("dw_general_res_off", (1, 16, 15, 15), (16, 1, 5, 5), dict(pads=4, dilation=2, groups=16), ("f32", "f16"),
     (1, 2, 3), True),
    # narrow depthwise kernel: x on 2 bytes only -> synchronous plane staging
    ("dw_narrow_half_off1", (2, 8, 14, 14), (8, 1, 5, 5), dict(pads=2, groups=8, act="hard_swish"),
     ("f16", "bf16"), (1, 1, 0), False),
    ("dw_narrow_f32_off3", (2, 8, 14, 14), (8, 1, 5, 5), dict(pads=2, groups=8, act="hard_swish"), ("f32",),
     (3, 1, 0), False),
    ("dw_narrow_odd_width", (2, 4, 9, 13), (4, 1, 3, 3), dict(pads=1, groups=4), ("f16",), (0, 0, 0), False),
    # CUDA-core pointwise without 16-byte B copies, scalar stores
    ("ffma_pointwise_off", (2, 16, 8, 8), (24, 16, 1, 1), dict(act="leaky_relu", alpha=0.1), ("f32",),
     (1, 2, 3), True),
    ("ffma_general_y_off", (1, 5, 19, 17), (20, 5, 4, 3), dict(stride=(1, 2), pads=(1, 1, 2, 0)), ("f32",),
     (2, 1, 1), True),
    # grouped CUDA-core layer with staged input rows, y and the residual off 4 bytes (scalar stores)
    ("grouped_y_off", (2, 32, 13, 12), (32, 16, 3, 3), dict(pads=2, dilation=2, groups=2, act="silu"), ("f32",),
     (0, 1, 1), True),
]


def _offset_params():
    out = []
    for case in OFFSET_CASES:
        for dt in case[4]:
            out.append(pytest.param(case, dt, id=f"{case[0]}-{dt}"))
    return out


@pytest.mark.parametrize("case,dtype", _offset_params())
def test_operands_at_element_offsets(case, dtype):
    name, xs, ws, g, _, offs, res = case
    p0 = conv.make_problem(xs, ws, dtype=dtype, has_bias=True, has_residual=res, **g)
    ho, wo = conv.conv_output_shape(p0)
    inp = random_layer_inputs(xs, ws, dtype, seed=len(name) * 31 + sum(offs), bias=True,
                              residual_shape=(xs[0], ws[0], ho, wo) if res else None)
    if name.startswith("window"):
        assert _desc(p0).startswith("igemm_tcgen05_window"), _desc(p0)
    if name.startswith("pw_"):
        assert _desc(p0).startswith("pointwise_mma"), _desc(p0)
    y, _ = _run_offsets(inp, dtype, offs, **g)
    out = check_full(inp, dtype, y, **g)
    assert out["ok"], out


def test_split_k_unaligned_output():
    xs, ws = (1, 512, 7, 7), (64, 512, 1, 1)
    inp = random_layer_inputs(xs, ws, "f32", seed=77, bias=True, residual_shape=(1, 64, 7, 7))
    p = conv.make_problem(xs, ws, dtype="f32", has_bias=True, has_residual=True)
    assert conv.conv_plan(p, torch.cuda.get_device_properties(0).multi_processor_count)["split_k"] > 1
    y, _ = _run_offsets(inp, "f32", (1, 3, 2))
    out = check_full(inp, "f32", y)
    assert out["ok"], out


# ---- chained layers ------------------------------------------------------
def _geo(L):
    return dict(stride=L.stride, pads=L.pads, dilation=L.dilation, groups=L.groups, act=L.act,
                alpha=L.alpha, beta=L.beta)


def _gpu_layer(L, x_dev, inp):
    """Run layer L on the device tensor x_dev with L's own weights / bias /
    residual from inp; returns y on the device."""
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items() if k != "x"}
    return conv.conv2d(x_dev, dev["w"], dev["bias"], dev["residual"], **_geo(L))


@pytest.mark.parametrize("first,second,size", [
    ("resnet50_3x3_f16", "resnet50_1x1_res_f16", (2, 24, 24)),
    ("resnet50_3x3_f16", "resnet50_1x1_res_f16", None),
    ("mbv3_dw5x5_f32", "mbv3_pw1x1_f32", (2, 28, 28)),
    ("mbv3_dw5x5_f16", "mbv3_pw1x1_f16", (2, 28, 28)),
    ("mbv3_dw5x5_f16", "mbv3_pw1x1_f16", None),
])
def test_chained_pair(first, second, size):
    """The second layer consumes the first layer's GPU output; both are
    checked against the oracle, the second on that very tensor."""
    A, B = LAYERS[first], LAYERS[second]
    assert B.feeds_from == A.name
    if size is not None:
        n, h, w = size
        A = dataclasses.replace(A, n=n, h=h, w=w)
        rs = (n, B.c_out, h, w) if B.residual_shape else None
        B = dataclasses.replace(B, n=n, h=h, w=w, residual_shape=rs)
    ia = make_inputs(A)
    ya = _gpu_layer(A, ia["x"].cuda(), ia)
    ib = make_inputs(B)
    yb = _gpu_layer(B, ya, ib)
    torch.cuda.synchronize()
    ib_chained = dict(ib, x=ya.cpu())
    if size is not None:
        ra = check_full(ia, A.dtype, ya.cpu(), **_geo(A))
        rb = check_full(ib_chained, B.dtype, yb.cpu(), **_geo(B))
    else:
        ra = check_sampled(ia, A.dtype, ya.cpu(), count=1500, seed=3, **_geo(A))
        rb = check_sampled(ib_chained, B.dtype, yb.cpu(), count=1500, seed=4, **_geo(B))
    assert ra["ok"], ra
    assert rb["ok"], rb


def test_unfolded_tail_split():
    """The CUDA-core kernel with its unfolded input and the last round of
    tiles split in k (a second kernel adds the ranges in order)."""
    xs, ws = (11, 32, 64, 64), (128, 32, 3, 3)
    g = dict(pads=1, act="silu")
    p = conv.make_problem(xs, ws, dtype="f32", has_bias=True, has_residual=True, **g)
    desc = conv.conv_describe_variant(p)
    assert "B=unfolded" in desc and "tail=" in desc and "launches=3" in desc, desc
    inp = random_layer_inputs(xs, ws, "f32", seed=91, bias=True, residual_shape=(11, 128, 64, 64))
    y, _ = _run_offsets(inp, "f32", (0, 0, 0), **g)
    out = check_full(inp, "f32", y, **g)
    assert out["ok"], out
    assert out["max_scaled_err"] < 1e-5, out
    y2, _ = _run_offsets(inp, "f32", (0, 0, 0), **g)
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))   # fixed order, no atomics


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("mode", ["SAME_UPPER", "SAME_LOWER", "VALID"])
@pytest.mark.parametrize("xs,ws,stride,dil", [
    ((2, 3, 37, 30), (8, 3, 7, 7), (2, 2), (1, 1)),
    ((1, 8, 20, 24), (16, 8, 4, 3), (1, 3), (2, 1)),
    ((2, 16, 9, 16), (16, 1, 5, 5), (1, 1), (1, 1)),
])
def test_auto_pad_convolution(dtype, mode, xs, ws, stride, dil):
    """ONNX auto_pad through the library against the oracle given the pads
    that the oracle's own auto_pad restatement computes."""
    from oracle import arith
    groups = xs[1] if ws[1] == 1 else 1
    dev = random_layer_inputs(xs, ws, dtype, seed=zlib.crc32(repr((mode, xs)).encode()) % 1000, bias=True)
    y = conv.conv2d(dev["x"].cuda(), dev["w"].cuda(), dev["bias"].cuda(), stride=stride, dilation=dil,
                    groups=groups, act="relu", auto_pad=mode)
    torch.cuda.synchronize()
    pt, pb = arith.auto_pad(xs[2], ws[2], stride[0], dil[0], mode)
    pl, pr = arith.auto_pad(xs[3], ws[3], stride[1], dil[1], mode)
    if mode != "VALID":
        assert tuple(y.shape[2:]) == (-(-xs[2] // stride[0]), -(-xs[3] // stride[1]))
    out = check_full(dev, dtype, y.cpu(), stride=stride, pads=(pt, pl, pb, pr), dilation=dil,
                     groups=groups, act="relu")
    assert out["ok"], out


# ---- batch chunking ----------------------------------------------------------
@pytest.mark.parametrize("xs,ws,g,dtype", [
    ((11, 32, 64, 64), (128, 32, 3, 3), dict(pads=1, act="silu"), "f32"),       # unfolded, tail split
    ((4, 256, 28, 28), (512, 256, 3, 3), dict(pads=1, act="relu"), "f32"),      # unfolded (Winograd off)
    ((5, 512, 7, 7), (64, 512, 1, 1), dict(act="leaky_relu", alpha=0.1), "f32"),  # split k, 49 px per image
    ((3, 256, 9, 9), (48, 256, 3, 3), dict(pads=1), "bf16"),                     # forced CUDA-core split k
])
def test_batch_chunks_are_bit_identical(xs, ws, g, dtype):
    """A scratch smaller than the whole batch needs (but at least one image's)
    runs the batch in chunks of whole images; the result has the same bits
    ("Convolution, pooling and resize", Layout and operands)."""
    flags = conv.FLAG_FORCE_FFMA if dtype != "f32" else conv.FLAG_NO_WINOGRAD
    p = conv.make_problem(xs, ws, dtype=dtype, has_bias=True, has_residual=True, flags=flags, **g)
    full = conv.conv_scratch_bytes(p)
    one = conv.conv_scratch_bytes_per_image(p)
    assert 0 < one < full, (one, full, conv.conv_describe_variant(p))
    ho, wo = conv.conv_output_shape(p)
    inp = random_layer_inputs(xs, ws, dtype, seed=xs[0] * 13 + ws[0], bias=True,
                              residual_shape=(xs[0], ws[0], ho, wo))
    dev = {k: v.cuda() for k, v in inp.items()}
    scratch = torch.empty(full, dtype=torch.uint8, device="cuda")

    def run(nbytes):
        y = torch.full((xs[0], ws[0], ho, wo), float("nan"), dtype=dev["x"].dtype, device="cuda")
        conv.conv_forward(p, dev["x"], dev["w"], dev["bias"], dev["residual"], y, scratch, nbytes)
        torch.cuda.synchronize()
        return y.cpu()

    def bits(y):
        return y.view(torch.int32 if y.dtype == torch.float32 else torch.int16)

    whole = run(full)
    out = check_full(inp, dtype, whole, **g)
    assert out["ok"], out
    for nbytes in (one, one + (full - one) // 3, full - 1):
        assert torch.equal(bits(run(nbytes)), bits(whole)), nbytes
    # less than one image's scratch is refused before anything runs
    lib = conv.load()
    y = torch.empty((xs[0], ws[0], ho, wo), dtype=dev["x"].dtype, device="cuda")
    st = lib.conv_forward(ctypes.byref(p), dev["x"].data_ptr(), dev["w"].data_ptr(), dev["bias"].data_ptr(),
                          dev["residual"].data_ptr(), y.data_ptr(), scratch.data_ptr(), one - 1, None)
    assert conv.STATUS[st] == "CONV_ERR_SCRATCH"


# ---- Winograd F(2x2, 3x3) ------------------------------------------------------
@pytest.mark.parametrize("xs,ws,g,res", [
    ((2, 8, 9, 11), (16, 8, 3, 3), dict(pads=1, act="relu"), True),
    ((1, 5, 12, 7), (6, 5, 3, 3), dict(pads=(2, 0, 1, 1), act="silu"), False),
    ((3, 4, 6, 6), (4, 4, 3, 3), dict(act="tanh"), True),                # no padding: 4x4 outputs
    ((1, 16, 1, 9), (8, 16, 3, 3), dict(pads=(1, 1, 1, 1)), False),       # one input row
    ((2, 64, 14, 14), (64, 64, 3, 3), dict(pads=1, act="leaky_relu", alpha=0.1), True),
])
def test_winograd_parity(xs, ws, g, res):
    """Winograd F(2x2, 3x3) against the oracle's direct sum: the float32 bar,
    literally (max |err| / sum|w x| < 1e-5)."""
    flags = conv.FLAG_WINOGRAD
    p = conv.make_problem(xs, ws, dtype="f32", has_bias=True, has_residual=res, flags=flags, **g)
    assert conv.conv_describe_variant(p).startswith("winograd_f2x2_3x3"), conv.conv_describe_variant(p)
    ho, wo = conv.conv_output_shape(p)
    inp = random_layer_inputs(xs, ws, "f32", seed=xs[1] * 7 + ws[0], bias=True,
                              residual_shape=(xs[0], ws[0], ho, wo) if res else None)
    y, _ = _run_offsets(inp, "f32", (0, 0, 0), flags=flags, **g)
    out = check_full(inp, "f32", y, **g)
    assert out["ok"], out
    assert out["max_scaled_err"] < 1e-5, out


# ---- host batches with the copies overlapped -------------------------------------
@pytest.mark.parametrize("dtype,xs,ws,geo,res", [
    ("f32", (2, 16, 18, 20), (24, 16, 3, 3), dict(pads=1, act="relu"), True),
    ("f16", (2, 16, 16, 16), (32, 16, 3, 3), dict(pads=1, act="silu"), False),
])
def test_host_pipeline_matches_conv2d(dtype, xs, ws, geo, res):
    """HostPipeline over five host batches gives, bit for bit, what conv2d
    gives on each batch (two device buffers in turn, three streams)."""
    tdt = {"f32": torch.float32, "f16": torch.float16}[dtype]
    w = random_layer_inputs(xs, ws, dtype, seed=5, bias=True)["w"].cuda()
    b = random_layer_inputs(xs, ws, dtype, seed=6, bias=True)["bias"].cuda()
    ho, wo = conv.conv_output_shape(conv.make_problem(xs, ws, dtype=dtype, **{k: v for k, v in geo.items() if k != "act"}))
    r = torch.randn((xs[0], ws[0], ho, wo), generator=torch.Generator().manual_seed(9)).to(tdt).cuda() if res else None
    xh = [torch.randn(xs, generator=torch.Generator().manual_seed(100 + i)).to(tdt).pin_memory() for i in range(5)]
    yh = [torch.empty((xs[0], ws[0], ho, wo), dtype=tdt).pin_memory() for _ in range(5)]
    pipe = conv.HostPipeline(xs, w, b, r, **geo)
    pipe.run(xh, yh)
    torch.cuda.synchronize()
    for i in range(5):
        ref = conv.conv2d(xh[i].cuda(), w, b, r, **geo)
        torch.cuda.synchronize()
        assert torch.equal(yh[i], ref.cpu()), i
