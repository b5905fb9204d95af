"""conv_forward_fixed_scratch: the forward call for callers that cannot
allocate device memory (a plug-in whose host framework owns all allocations,
a path that must not enter the allocator).  Its split-k planes live in the
library's own fixed device array instead of caller scratch.

This file is collected last on purpose: it checks the fixed array against the
ordinary entry point on a layer that needs scratch, twice in a row (the second
call finds the first call's leftovers in the array), and that a problem too
large for the array is refused before anything runs.
"""
import ctypes

import numpy as np
import pytest
import torch

import implicit_gemm_cnn_gb300 as conv
from gpu_util import oracle_ref
from oracle.parity import compare
from workloads import LAYERS, make_inputs, to_numpy_operand

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _problem(L, flags=0):
    return conv.make_problem((L.n, L.c_in, L.h, L.w), (L.c_out, L.c_in // L.groups, L.kh, L.kw),
                             dtype=L.dtype, stride=L.stride, pads=L.pads, dilation=L.dilation,
                             groups=L.groups, act=L.act, alpha=L.alpha, beta=L.beta,
                             has_bias=L.bias, has_residual=L.residual_shape is not None, flags=flags)


def test_fixed_scratch_matches_conv_forward_twice():
    L = LAYERS["late_1x1_splitk_f32"]          # a layer whose plan splits k into scratch planes
    p = _problem(L)
    need = conv.conv_scratch_bytes(p)
    assert 0 < need <= conv.FIXED_SCRATCH_BYTES
    inp = make_inputs(L)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ho, wo = conv.conv_output_shape(p)
    shape = (L.n, L.c_out, ho, wo)
    # the existing entry point, with caller-provided scratch
    y_ref = torch.empty(shape, dtype=dev["x"].dtype, device="cuda")
    scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    conv.conv_forward(p, dev["x"], dev["w"], dev["bias"], dev["residual"], y_ref, scratch, need)
    torch.cuda.synchronize()
    ref = oracle_ref(inp, L.dtype, stride=L.stride, pads=L.pads, dilation=L.dilation,
                     groups=L.groups, act=L.act, alpha=L.alpha, beta=L.beta)
    ref["y"] = to_numpy_operand(y_ref.cpu(), L.dtype)   # compare against the existing entry point
    for call in range(2):
        y = torch.full(shape, float("nan"), dtype=dev["x"].dtype, device="cuda")
        conv.conv_forward_fixed_scratch(p, dev["x"], dev["w"], dev["bias"], dev["residual"], y)
        torch.cuda.synchronize()
        got = to_numpy_operand(y.cpu(), L.dtype)
        res = compare(got, ref, L.dtype, L.act, L.alpha, L.beta,
                      bias=to_numpy_operand(inp["bias"], L.dtype))
        assert res["ok"], (call, res)
        assert np.array_equal(got, ref["y"]), call      # same kernels, same summation order


def test_fixed_scratch_refuses_oversize_problems():
    # a forced 40-way split of a 2048 x 32 x 32 output needs 40 * 2M * 4 B = 320 MiB of planes
    p = conv.make_problem((1, 256, 32, 32), (2048, 256, 1, 1), dtype="f32",
                          flags=conv.FLAG_FORCE_FFMA | (40 << conv.SPLIT_K_SHIFT))
    assert conv.conv_scratch_bytes(p) > conv.FIXED_SCRATCH_BYTES
    lib = conv.load()
    fake = ctypes.c_void_p(0x1000)   # refused before any pointer is used or anything is enqueued
    status = lib.conv_forward_fixed_scratch(ctypes.byref(p), fake, fake, None, None, fake, None)
    assert conv.STATUS[status] == "CONV_ERR_SCRATCH"
