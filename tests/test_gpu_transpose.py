"""The transposed convolution on the GPU against the CPU oracle, element by
element, with the parity bar of the forward convolution ("Convolution,
pooling and resize", Tolerances: Conv and ConvTranspose share 1e-5 / 2e-3)."""
import dataclasses
import zlib

import numpy as np
import pytest
import torch

import implicit_gemm_cnn_gb300 as conv
from gpu_util import orc
from oracle.parity import compare
from workloads import TRANSPOSE_LAYERS, make_transpose_inputs, random_layer_inputs, to_numpy_operand

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _run(inp, **g):
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y = conv.conv_transpose2d(dev["x"], dev["w"], dev.get("bias"), dev.get("residual"), **g)
    torch.cuda.synchronize()
    return y.cpu()


def _check(inp, dtype, y, index=None, **g):
    st, dl, op = conv._pair(g.get("stride", 1)), conv._pair(g.get("dilation", 1)), conv._pair(g.get("out_pad", 0))
    ops = [to_numpy_operand(inp.get(k), dtype) for k in ("x", "w", "bias", "residual")]
    ref = orc().conv_transpose2d(*ops, dtype=dtype, stride=st, pads=conv._pads(g.get("pads", 0)), dilation=dl,
                                 out_pad=op, groups=g.get("groups", 1), act=g.get("act", "identity"),
                                 alpha=g.get("alpha", 0.0), beta=g.get("beta", 0.0), index=index)
    yn = to_numpy_operand(y, dtype)
    res = None
    if index is not None:
        yn = yn.reshape(-1)[index]
        c, hw = y.shape[1], y.shape[2] * y.shape[3]
        co = (index // hw) % c
        res_s = to_numpy_operand(inp["residual"], dtype).reshape(-1)[index] if inp.get("residual") is not None else None
        return compare(yn, ref, dtype, g.get("act", "identity"), g.get("alpha", 0.0), g.get("beta", 0.0),
                       bias=ops[2], residual=res_s, co_index=co)
    return compare(yn, ref, dtype, g.get("act", "identity"), g.get("alpha", 0.0), g.get("beta", 0.0),
                   bias=ops[2], residual=ops[3])


# (name, x shape, w shape [Cin][Cout/g][kh][kw], geometry, residual)
CASES = [
    ("s2_k3_p1_op1", (2, 8, 7, 6), (8, 5, 3, 3), dict(stride=2, pads=1, out_pad=1, act="relu"), False),
    ("s2_k4_uniform", (2, 16, 9, 8), (16, 8, 4, 4), dict(stride=2, pads=1, act="silu"), True),
    ("s2_k2_unet", (1, 12, 10, 10), (12, 6, 2, 2), dict(stride=2), False),
    ("s3_dil2_asym", (1, 6, 8, 7), (6, 4, 3, 2), dict(stride=(3, 2), pads=(2, 1, 0, 2), dilation=(2, 1),
                                                      out_pad=(1, 0), act="leaky_relu", alpha=0.1), True),
    ("grouped", (2, 12, 6, 9), (12, 3, 3, 3), dict(stride=2, pads=1, groups=4, act="tanh"), False),
    ("s1_same", (1, 10, 11, 12), (10, 7, 3, 3), dict(pads=1, act="hard_swish"), True),
    ("one_d", (3, 8, 1, 20), (8, 4, 1, 5), dict(stride=(1, 3), pads=(0, 2, 0, 1), out_pad=(0, 2)), False),
]


def _case_params():
    """Every case in every element type; 16-bit types also with the Gemm kept
    on the CUDA cores (the tensor-core Gemm is the default for one group)."""
    out = []
    for c in CASES:
        for dt in ("f32", "f16", "bf16"):
            out.append(pytest.param(c, dt, 0, id=f"{c[0]}-{dt}"))
            if dt != "f32":
                out.append(pytest.param(c, dt, conv.FLAG_NO_PW_MMA, id=f"{c[0]}-{dt}-cudacore"))
    return out


@pytest.mark.parametrize("case,dtype,flags", _case_params())
def test_transpose_cases(case, dtype, flags):
    name, xs, ws, g, res = case
    g = dict(g, flags=flags) if flags else g
    p = conv.make_transpose_problem(xs, ws, dtype=dtype, has_bias=True, has_residual=res,
                                    **{k: v for k, v in g.items() if k not in ("act", "alpha", "beta", "flags")})
    ho, wo = conv.conv_transpose_output_shape(p)
    cout = ws[1] * g.get("groups", 1)
    seed = zlib.crc32(name.encode()) % 1000
    inp = random_layer_inputs(xs, ws, dtype, seed=seed, bias=False)
    gen = torch.Generator().manual_seed(seed + 1)
    dt = inp["x"].dtype
    inp["bias"] = (torch.rand((cout,), generator=gen) * 2 - 1).to(dt)
    inp["residual"] = (torch.rand((xs[0], cout, ho, wo), generator=gen) * 2 - 1).to(dt) if res else None
    y = _run(inp, **g)
    assert tuple(y.shape) == (xs[0], cout, ho, wo)
    out = _check(inp, dtype, y, **g)
    assert out["ok"], out
    if dtype == "f32":
        assert out["max_scaled_err"] < 1e-5, out


@pytest.mark.parametrize("name", sorted(TRANSPOSE_LAYERS))
def test_transpose_layer_reduced_all_outputs(name):
    L = dataclasses.replace(TRANSPOSE_LAYERS[name], n=1, h=10, w=12)
    inp = make_transpose_inputs(L)
    g = dict(stride=L.stride, pads=L.pads, dilation=L.dilation, out_pad=L.out_pad, groups=L.groups, act=L.act)
    out = _check(inp, L.dtype, _run(inp, **g), **g)
    assert out["ok"], out


@pytest.mark.parametrize("name", sorted(TRANSPOSE_LAYERS))
def test_transpose_layer_full_size_sampled(name):
    L = TRANSPOSE_LAYERS[name]
    inp = make_transpose_inputs(L)
    g = dict(stride=L.stride, pads=L.pads, dilation=L.dilation, out_pad=L.out_pad, groups=L.groups, act=L.act)
    y = _run(inp, **g)
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.integers(0, y.numel(), 2500), [0, y.numel() - 1]])).astype(np.int64)
    out = _check(inp, L.dtype, y, index=idx, **g)
    assert out["ok"], out
    y2 = _run(inp, **g)
    assert torch.equal(y.view(torch.int16 if y.dtype != torch.float32 else torch.int32),
                       y2.view(torch.int16 if y2.dtype != torch.float32 else torch.int32))
