"""Helpers of the GPU parity tests: run the library through its C ABI, run the
oracle on the same inputs, compare with the parity bar."""
from __future__ import annotations

import numpy as np
import torch

import implicit_gemm_cnn_gb300 as conv
import oracle
from oracle.parity import compare
from workloads import to_numpy_operand

_ORACLE = None


def orc():
    global _ORACLE
    if _ORACLE is None:
        _ORACLE = oracle.Oracle()
    return _ORACLE


def geometry(**g):
    return dict(stride=g.get("stride", 1), pads=g.get("pads", 0), dilation=g.get("dilation", 1),
                groups=g.get("groups", 1), act=g.get("act", "identity"),
                alpha=g.get("alpha", 0.0), beta=g.get("beta", 0.0))


def run_gpu(inp: dict, flags: int = 0, **g) -> torch.Tensor:
    dev = torch.device("cuda")
    x = inp["x"].to(dev)
    w = inp["w"].to(dev)
    b = inp["bias"].to(dev) if inp.get("bias") is not None else None
    r = inp["residual"].to(dev) if inp.get("residual") is not None else None
    y = conv.conv2d(x, w, b, r, flags=flags, **geometry(**g))
    torch.cuda.synchronize()
    return y.cpu()


def _oracle_args(g):
    gg = geometry(**g)
    st = conv._pair(gg["stride"])
    dl = conv._pair(gg["dilation"])
    pads = conv._pads(gg["pads"])
    return dict(stride=st, pads=pads, dilation=dl, groups=gg["groups"], act=gg["act"],
                alpha=gg["alpha"], beta=gg["beta"])


def oracle_ref(inp: dict, dtype: str, index=None, **g) -> dict:
    ops = [to_numpy_operand(inp.get(k), dtype) for k in ("x", "w", "bias", "residual")]
    return orc().conv2d(*ops, dtype=dtype, index=index, **_oracle_args(g))


def check_full(inp: dict, dtype: str, y: torch.Tensor, **g) -> dict:
    ref = oracle_ref(inp, dtype, **g)
    yn = to_numpy_operand(y, dtype)
    res = compare(yn, ref, dtype, geometry(**g)["act"], geometry(**g)["alpha"],
                  geometry(**g)["beta"], bias=to_numpy_operand(inp.get("bias"), dtype),
                  residual=to_numpy_operand(inp.get("residual"), dtype))
    return res


def sample_indices(shape, count: int, seed: int) -> np.ndarray:
    """Random NCHW output indices plus every corner / edge class: first and
    last image, channel, row and column."""
    n, c, h, w = shape
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, n * c * h * w, count).tolist())
    for nn in {0, n - 1}:
        for cc in {0, c // 2, c - 1}:
            for hh in {0, 1, h // 2, h - 2 if h > 1 else 0, h - 1}:
                for ww in {0, 1, w // 2, w - 2 if w > 1 else 0, w - 1}:
                    idx.add(((nn * c + cc) * h + hh) * w + ww)
    return np.array(sorted(idx), dtype=np.int64)


def check_sampled(inp: dict, dtype: str, y: torch.Tensor, count: int = 3000, seed: int = 0, **g):
    shape = tuple(y.shape)
    idx = sample_indices(shape, count, seed)
    ref = oracle_ref(inp, dtype, index=idx, **g)
    yn = to_numpy_operand(y, dtype).reshape(-1)[idx]
    c, hw = shape[1], shape[2] * shape[3]
    co = (idx // hw) % c
    res_s = None
    if inp.get("residual") is not None:
        res_s = to_numpy_operand(inp["residual"], dtype).reshape(-1)[idx]
    gg = geometry(**g)
    return compare(yn, ref, dtype, gg["act"], gg["alpha"], gg["beta"],
                   bias=to_numpy_operand(inp.get("bias"), dtype), residual=res_s, co_index=co)
