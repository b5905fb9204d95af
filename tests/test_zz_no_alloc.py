"""conv_forward_fixed_scratch: the forward call for callers that cannot
allocate device memory (a plug-in whose host framework owns all allocations,
a path that must not enter the allocator).  Its scratch -- split-k planes,
the shifted-window kernel's repacked weights, the CUDA-core kernel's
unfolded input, Winograd's transformed operands -- lives in the library's own
fixed device array instead of caller memory.

This file is collected last on purpose.  Every call here is compared bit for
bit with the ordinary entry point on the same inputs, and calls alternate
between problems and inputs, so the array always holds another call's data
when a call starts: a byte a call reads without writing it first would show.
A problem whose scratch does not fit the array runs on a variant that needs
none (checked against conv_forward with that variant forced), and a forced
split that does not fit is refused before anything runs.
"""
import ctypes

import numpy as np
import pytest
import torch

import implicit_gemm_cnn_gb300 as conv
from gpu_util import check_full
from workloads import random_layer_inputs, to_numpy_operand

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _case(xs, ws, dtype, seed, flags=0, **g):
    p = conv.make_problem(xs, ws, dtype=dtype, has_bias=True, flags=flags, **g)
    inp = random_layer_inputs(xs, ws, dtype, seed=seed, bias=True)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    return p, inp, dev, g


def _ordinary(p, dev, extra_flags=0):
    """y from conv_forward with caller scratch (and optionally a forced variant)."""
    q = conv.ConvProblem.from_buffer_copy(p)
    q.flags |= extra_flags
    ho, wo = conv.conv_output_shape(q)
    y = torch.empty((q.n, q.c_out, ho, wo), dtype=dev["x"].dtype, device="cuda")
    need = conv.conv_scratch_bytes(q)
    scratch = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    conv.conv_forward(q, dev["x"], dev["w"], dev["bias"], None, y, scratch if need else None, need)
    torch.cuda.synchronize()
    return y


def _fixed(p, dev):
    ho, wo = conv.conv_output_shape(p)
    y = torch.full((p.n, p.c_out, ho, wo), float("nan"), dtype=dev["x"].dtype, device="cuda")
    conv.conv_forward_fixed_scratch(p, dev["x"], dev["w"], dev["bias"], None, y)
    torch.cuda.synchronize()
    return y


def _bits(y):
    return y.view(torch.int32 if y.dtype == torch.float32 else torch.int16).cpu()


def _check(case, extra_flags=0):
    p, inp, dev, g = case
    want = _ordinary(p, dev, extra_flags)
    got = _fixed(p, dev)
    assert torch.equal(_bits(got), _bits(want))
    dt = {0: "f32", 1: "f16", 2: "bf16"}[p.dtype]
    res = check_full(inp, dt, got.cpu(), **g)
    assert res["ok"], res


def test_fixed_scratch_split_k_alternating_inputs():
    """Split-k planes in the array (the planes form of the split, forced by
    CONV_FLAG_NO_CLUSTER_K): calls alternating between two shapes and values,
    each equal to conv_forward's bits; then the default form, whose ranges
    are reduced within a thread-block cluster and leave the array unread."""
    a = _case((1, 2048, 7, 7), (512, 2048, 1, 1), "f32", seed=41, flags=conv.FLAG_NO_CLUSTER_K)
    b = _case((1, 1024, 9, 9), (96, 1024, 3, 3), "f32", seed=42,
              flags=conv.FLAG_NO_WINOGRAD | conv.FLAG_NO_CLUSTER_K, pads=1, act="relu")
    a_cluster = _case((1, 2048, 7, 7), (512, 2048, 1, 1), "f32", seed=49)
    for c in (a, b, a_cluster):
        assert conv.conv_plan(c[0], torch.cuda.get_device_properties(0).multi_processor_count)["split_k"] > 1
        assert 0 < conv.conv_scratch_bytes(c[0]) <= conv.FIXED_SCRATCH_BYTES
    assert "reduce=planes" in conv.conv_describe_variant(a[0])
    assert "reduce=cluster" in conv.conv_describe_variant(a_cluster[0])
    for c in (a, b, a, a_cluster, b):
        _check(c)


def test_fixed_scratch_shifted_window_alternating_layers():
    """Repacked weights of the shifted-window kernel in the array: a 3x3 layer,
    a stride-2 7x7 layer, the 3x3 layer again with other weights."""
    a = _case((2, 64, 24, 24), (64, 64, 3, 3), "f16", seed=43, pads=1, act="relu")
    b = _case((2, 3, 48, 48), (64, 3, 7, 7), "f16", seed=44, stride=2, pads=3, act="relu")
    a2 = _case((2, 64, 24, 24), (64, 64, 3, 3), "f16", seed=45, pads=1, act="relu")
    for c in (a, b):
        assert conv.conv_describe_variant(c[0]).startswith("igemm_tcgen05_window")
        assert 0 < conv.conv_scratch_bytes(c[0]) <= conv.FIXED_SCRATCH_BYTES
    for c in (a, b, a2, b):
        _check(c)


def test_fixed_scratch_window_too_large_runs_gather_variant():
    """Repacked weights past the array: the gather tensor-core kernel, which
    needs no scratch, runs the problem instead of a refusal."""
    c = _case((1, 64, 16, 16), (8192, 64, 3, 3), "bf16", seed=46, pads=1)
    p = c[0]
    assert conv.conv_describe_variant(p).startswith("igemm_tcgen05_window")
    assert conv.conv_scratch_bytes(p) > conv.FIXED_SCRATCH_BYTES
    _check(c, extra_flags=conv.FLAG_NO_WINDOW)


def test_fixed_scratch_split_too_large_runs_unsplit():
    """An automatic split whose planes exceed the array runs k in one range."""
    c = _case((1, 2048, 16, 16), (4096, 2048, 1, 1), "f32", seed=47)
    p = c[0]
    assert conv.conv_scratch_bytes(p) > conv.FIXED_SCRATCH_BYTES
    _check(c, extra_flags=conv.FLAG_NO_SPLIT_K)


def test_fixed_scratch_unfolded_too_large_runs_gathered():
    """The CUDA-core kernel's unfolded input copy past the array: the same
    kernel with its B operand gathered from x, which needs no scratch."""
    c = _case((4, 256, 28, 28), (512, 256, 3, 3), "f32", seed=48, flags=conv.FLAG_NO_WINOGRAD, pads=1, act="relu")
    p = c[0]
    assert "B=unfolded" in conv.conv_describe_variant(p)
    assert conv.conv_scratch_bytes(p) > conv.FIXED_SCRATCH_BYTES
    _check(c, extra_flags=conv.FLAG_NO_UNFOLD)


def test_fixed_scratch_winograd_too_large_runs_direct():
    """Winograd's transformed operands past the array: the direct CUDA-core
    kernel with its input gathered from x, which needs no scratch."""
    c = _case((4, 256, 28, 28), (512, 256, 3, 3), "f32", seed=49, pads=1, act="relu")
    p = c[0]
    assert conv.conv_describe_variant(p).startswith("winograd_f2x2_3x3")
    assert conv.conv_scratch_bytes(p) > conv.FIXED_SCRATCH_BYTES
    _check(c, extra_flags=conv.FLAG_NO_WINOGRAD | conv.FLAG_NO_UNFOLD)


def test_fixed_scratch_refuses_oversize_forced_split():
    # a forced 40-way split of a 2048 x 32 x 32 output needs 40 * 2M * 4 B = 320 MiB of planes
    p = conv.make_problem((1, 256, 32, 32), (2048, 256, 1, 1), dtype="f32",
                          flags=conv.FLAG_FORCE_FFMA | (40 << conv.SPLIT_K_SHIFT))
    assert conv.conv_scratch_bytes(p) > conv.FIXED_SCRATCH_BYTES
    lib = conv.load()
    fake = ctypes.c_void_p(0x1000)   # refused before any pointer is used or anything is enqueued
    status = lib.conv_forward_fixed_scratch(ctypes.byref(p), fake, fake, None, None, fake, None)
    assert conv.STATUS[status] == "CONV_ERR_SCRATCH"
