"""Seeded synthetic inputs for the convolution layers that are tested and timed.

This module is shared by the tests, the benchmark and the smoke check.  It
holds layer descriptions (shapes, pads, activation, element type, the value
distributions) and seeded generators -- and none of the convolution's
arithmetic: output shapes that a layer needs (the residual's) are written out
from the layer description, not computed here.

The layers are the vision workloads the convolution is measured on:
ResNet-50 (stem; 3x3 then 1x1-with-residual bottleneck pair), a
MobileNetV3-style block (5x5 depthwise then 1x1 pointwise), a grouped /
dilated / small-grid fp32 set, and one small fp32 layer.  Values are drawn
with ``torch.Generator`` on the CPU from a per-layer seed, in float32, then
rounded to the element type; every consumer reads the rounded values.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Layer:
    name: str
    n: int
    c_in: int
    h: int
    w: int
    c_out: int
    kh: int
    kw: int
    stride: tuple = (1, 1)
    pads: tuple = (0, 0, 0, 0)          # ONNX order: top, left, bottom, right
    dilation: tuple = (1, 1)
    groups: int = 1
    act: str = "identity"
    alpha: float = 0.0
    beta: float = 0.0
    dtype: str = "f32"                  # "f32", "f16", "bf16"
    bias: bool = True
    residual_shape: tuple | None = None  # (N, Cout, Ho, Wo) when a residual is added
    x_dist: tuple = ("uniform", -1.0, 1.0)
    w_dist: tuple = ("uniform", -1.0, 1.0)
    b_dist: tuple = ("uniform", -1.0, 1.0)
    r_dist: tuple = ("normal", 0.0, 1.0)
    seed: int = 0
    feeds_from: str | None = None       # the layer whose output is this layer's input
    description: str = ""

    def with_(self, **kw) -> "Layer":
        return dataclasses.replace(self, **kw)


def _he(fan_in: int) -> tuple:
    return ("normal", 0.0, math.sqrt(2.0 / fan_in))


LAYERS: dict[str, Layer] = {}


def _add(layer: Layer) -> None:
    LAYERS[layer.name] = layer


# Small fp32 layer (also the case the oracle finishes in well under a second).
_add(Layer("small_3x3_f32", 1, 3, 32, 32, 16, 3, 3, pads=(1, 1, 1, 1), act="relu",
           seed=1000, description="N=1 3->16 3x3 s1 p1 on 32x32, bias, ReLU, fp32"))
# ResNet-50 stem.
_add(Layer("resnet50_stem_f16", 8, 3, 224, 224, 64, 7, 7, stride=(2, 2), pads=(3, 3, 3, 3),
           act="relu", dtype="f16", x_dist=("normal", 0.0, 1.0), w_dist=_he(3 * 49),
           b_dist=("uniform", -0.1, 0.1), seed=1001,
           description="ResNet-50 stem: N=8 3->64 7x7 s2 p3, 224->112, bias, ReLU, fp16"))
# ResNet-50 bottleneck pair at N=32, 56x56.
_add(Layer("resnet50_3x3_f16", 32, 64, 56, 56, 64, 3, 3, pads=(1, 1, 1, 1), act="relu",
           dtype="f16", x_dist=("normal", 0.0, 1.0), w_dist=_he(64 * 9),
           b_dist=("uniform", -0.1, 0.1), seed=1002,
           description="ResNet-50 bottleneck 3x3 64->64 s1 p1 at 56x56, N=32, bias, ReLU, fp16"))
_add(Layer("resnet50_1x1_res_f16", 32, 64, 56, 56, 256, 1, 1, act="relu", dtype="f16",
           residual_shape=(32, 256, 56, 56), x_dist=("normal", 0.0, 1.0), w_dist=_he(64),
           b_dist=("uniform", -0.1, 0.1), r_dist=("normal", 0.0, 1.0), seed=1003,
           feeds_from="resnet50_3x3_f16",
           description="ResNet-50 bottleneck 1x1 64->256 at 56x56, N=32, bias + residual + ReLU, fp16"))
# MobileNetV3-style block at N=32, C=240, 28x28 (fp32 and fp16).
for _dt, _s in (("f32", 1004), ("f16", 1005)):
    _add(Layer(f"mbv3_dw5x5_{_dt}", 32, 240, 28, 28, 240, 5, 5, pads=(2, 2, 2, 2), groups=240,
               act="hard_swish", dtype=_dt, x_dist=("uniform", 0.0, 1.0), w_dist=_he(25),
               b_dist=("uniform", -0.1, 0.1), seed=_s,
               description=f"MobileNetV3 depthwise 5x5 C=240 g=240 p2 at 28x28, N=32, bias, hard-swish, {_dt}"))
    _add(Layer(f"mbv3_pw1x1_{_dt}", 32, 240, 28, 28, 40, 1, 1, act="identity", dtype=_dt,
               x_dist=("uniform", 0.0, 1.0), w_dist=_he(240), b_dist=("uniform", -0.1, 0.1),
               seed=_s + 2, feeds_from=f"mbv3_dw5x5_{_dt}",
               description=f"MobileNetV3 pointwise 1x1 240->40 at 28x28, N=32, bias, identity, {_dt}"))
# Grouped / dilated / small-grid fp32 set, all values U(-1, 1).
_add(Layer("grouped_dil2_f32", 16, 512, 28, 28, 512, 3, 3, pads=(2, 2, 2, 2), dilation=(2, 2),
           groups=32, act="silu", seed=1008,
           description="N=16 512->512 3x3 dilation 2 pad 2 groups 32 at 28x28, bias, SiLU, fp32"))
_add(Layer("late_1x1_splitk_f32", 1, 2048, 7, 7, 512, 1, 1, act="identity", seed=1009,
           description="N=1 2048->512 1x1 at 7x7 (split-k), bias, fp32"))
_add(Layer("strided_3x3_s2_f32", 16, 256, 56, 56, 512, 3, 3, stride=(2, 2), pads=(1, 1, 1, 1),
           act="leaky_relu", alpha=0.1, bias=False, seed=1010,
           description="N=16 256->512 3x3 s2 p1 at 56x56, leaky-relu 0.1, no bias, fp32"))

# A ResNet-50 stage-3 3x3 layer in float32: the stride-1 3x3 class on which
# "Convolution, pooling and resize" prices Winograd F(2x2, 3x3).
_add(Layer("resnet50_3x3_256_f32", 16, 256, 14, 14, 256, 3, 3, pads=(1, 1, 1, 1), act="relu",
           x_dist=("normal", 0.0, 1.0), w_dist=_he(256 * 9), b_dist=("uniform", -0.1, 0.1), seed=1011,
           description="ResNet-50 3x3 256->256 s1 p1 at 14x14, N=16, bias, ReLU, fp32"))

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _draw(shape, dist, gen) -> torch.Tensor:
    kind, a, b = dist
    if kind == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * (b - a) + a
    if kind == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * b + a
    raise ValueError(kind)


def make_inputs(layer: Layer, seed_offset: int = 0) -> dict:
    """CPU torch tensors (x, w, bias or None, residual or None) in the layer's
    element type, drawn from the layer's seed (+ ``seed_offset`` for extra,
    distinct sets of the same shape)."""
    gen = torch.Generator().manual_seed(layer.seed * 1000 + seed_offset)
    dt = TORCH_DTYPE[layer.dtype]
    x = _draw((layer.n, layer.c_in, layer.h, layer.w), layer.x_dist, gen).to(dt)
    w = _draw((layer.c_out, layer.c_in // layer.groups, layer.kh, layer.kw), layer.w_dist, gen).to(dt)
    b = _draw((layer.c_out,), layer.b_dist, gen).to(dt) if layer.bias else None
    r = _draw(layer.residual_shape, layer.r_dist, gen).to(dt) if layer.residual_shape else None
    return {"x": x, "w": w, "bias": b, "residual": r}


def random_layer_inputs(shape_x, shape_w, dtype: str, seed: int, bias=True,
                        residual_shape=None, dist=("uniform", -1.0, 1.0)) -> dict:
    """Inputs for an ad-hoc test shape, all from one distribution."""
    gen = torch.Generator().manual_seed(seed)
    dt = TORCH_DTYPE[dtype]
    x = _draw(tuple(shape_x), dist, gen).to(dt)
    w = _draw(tuple(shape_w), dist, gen).to(dt)
    b = _draw((shape_w[0],), dist, gen).to(dt) if bias else None
    r = _draw(tuple(residual_shape), dist, gen).to(dt) if residual_shape else None
    return {"x": x, "w": w, "bias": b, "residual": r}


def to_numpy_operand(t: torch.Tensor | None, dtype: str):
    """A CPU tensor as the numpy array the oracle reads: float32 values, or the
    uint16 bit patterns of a half / bfloat16 tensor."""
    if t is None:
        return None
    t = t.detach().cpu().contiguous()
    if dtype == "f32":
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


# ---- ConvInteger layers ------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class IntLayer:
    """A ConvInteger layer: uint8 / int8 operands, zero points, int32 output."""
    name: str
    n: int
    c_in: int
    h: int
    w: int
    c_out: int
    kh: int
    kw: int
    stride: tuple = (1, 1)
    pads: tuple = (0, 0, 0, 0)
    dilation: tuple = (1, 1)
    groups: int = 1
    x_type: str = "u8"
    w_type: str = "i8"
    per_channel: bool = True      # one weight zero point per output channel
    seed: int = 0
    description: str = ""

    def with_(self, **kw) -> "IntLayer":
        return dataclasses.replace(self, **kw)


INT_LAYERS: dict[str, IntLayer] = {}
# the second convolution of a Whisper-small-like audio front end (1-D as
# height 1): 768 -> 768 channels, kernel 3, stride 2, over 3000 frames, batch 8
INT_LAYERS["whisper_conv2_u8i8"] = IntLayer(
    "whisper_conv2_u8i8", 8, 768, 1, 3000, 768, 1, 3, stride=(1, 2), pads=(0, 1, 0, 1), seed=1100,
    description="ConvInteger 768->768 1x3 stride 2 over 3000 frames (1-D), N=8, uint8 x, int8 w, "
                "per-channel weight zero points")

_INT_RANGE = {"u8": (0, 256, torch.uint8), "i8": (-128, 128, torch.int8)}


def make_int_inputs(layer: IntLayer, seed_offset: int = 0) -> dict:
    """CPU tensors x, w (uniform over their type), x_zero (one value) and
    w_zero (one per output channel, within +-8 of zero, or one value)."""
    gen = torch.Generator().manual_seed(layer.seed * 1000 + seed_offset)
    xl, xh, xt = _INT_RANGE[layer.x_type]
    wl, wh, wt = _INT_RANGE[layer.w_type]
    x = torch.randint(xl, xh, (layer.n, layer.c_in, layer.h, layer.w), generator=gen).to(xt)
    w = torch.randint(wl, wh, (layer.c_out, layer.c_in // layer.groups, layer.kh, layer.kw), generator=gen).to(wt)
    xz = torch.randint(xl, xh, (1,), generator=gen).to(xt)
    nz = layer.c_out if layer.per_channel else 1
    wz = torch.randint(max(wl, -8), min(wh, 9), (nz,), generator=gen).to(wt)
    return {"x": x, "w": w, "x_zero": xz, "w_zero": wz}


# ---- transposed convolution layers ---------------------------------------------
@dataclasses.dataclass(frozen=True)
class TransposeLayer:
    """A ConvTranspose layer: w is [Cin][Cout/groups][kh][kw]."""
    name: str
    n: int
    c_in: int
    h: int
    w: int
    c_out: int
    kh: int
    kw: int
    stride: tuple = (1, 1)
    pads: tuple = (0, 0, 0, 0)
    dilation: tuple = (1, 1)
    out_pad: tuple = (0, 0)
    groups: int = 1
    act: str = "identity"
    dtype: str = "f32"
    bias: bool = True
    seed: int = 0
    description: str = ""


TRANSPOSE_LAYERS: dict[str, TransposeLayer] = {}
for _dt, _s in (("f32", 1200), ("f16", 1201)):
    # a decoder's 2x upsampling step: k = 2s gives every output the same
    # number of taps ("Convolutions", section 2.5)
    TRANSPOSE_LAYERS[f"decoder_up4x4_s2_{_dt}"] = TransposeLayer(
        f"decoder_up4x4_s2_{_dt}", 8, 256, 28, 28, 128, 4, 4, stride=(2, 2), pads=(1, 1, 1, 1), act="relu",
        dtype=_dt, seed=_s,
        description=f"ConvTranspose 256->128 4x4 stride 2 pad 1, 28x28 -> 56x56, N=8, bias, ReLU, {_dt}")


def make_transpose_inputs(layer: TransposeLayer, seed_offset: int = 0) -> dict:
    """x ~ U(-1, 1), w ~ N(0, sqrt(2 / fan_in)) with fan_in = Cin/groups * k^2
    / stride^2 (the taps that reach one output), bias ~ U(-0.1, 0.1)."""
    gen = torch.Generator().manual_seed(layer.seed * 1000 + seed_offset)
    dt = TORCH_DTYPE[layer.dtype]
    fan = (layer.c_in // layer.groups) * layer.kh * layer.kw / (layer.stride[0] * layer.stride[1])
    x = _draw((layer.n, layer.c_in, layer.h, layer.w), ("uniform", -1.0, 1.0), gen).to(dt)
    w = _draw((layer.c_in, layer.c_out // layer.groups, layer.kh, layer.kw), ("normal", 0.0, math.sqrt(2.0 / fan)),
              gen).to(dt)
    b = _draw((layer.c_out,), ("uniform", -0.1, 0.1), gen).to(dt) if layer.bias else None
    return {"x": x, "w": w, "bias": b, "residual": None}
