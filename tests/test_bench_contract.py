"""The arithmetic behind bench.py's JSON line, on the host: per-layer FLOPs and
algorithmic bytes against closed forms, the binding roofline each workload
layer is reported against, the whole-job rate and the rule that a committed
ncu summary's traffic only counts while its kernel source is unchanged."""
import dataclasses
import hashlib
import os

import bench
from workloads import LAYERS


def test_flops_closed_forms():
    # ResNet-50 stem: 2 * 8 * 112 * 112 * 64 * 3 * 7 * 7 (MACs Ho*Wo*Co*Ci*k^2/g per image, x2)
    assert bench.layer_flops(LAYERS["resnet50_stem_f16"]) == 2 * 8 * 112 * 112 * 64 * 3 * 49
    # grouped: 32 groups of 16 -> 16 channels, dilation 2 keeps 28 x 28
    assert bench.layer_flops(LAYERS["grouped_dil2_f32"]) == 2 * 16 * 28 * 28 * 512 * 16 * 9
    # depthwise: one input channel per output channel
    assert bench.layer_flops(LAYERS["mbv3_dw5x5_f32"]) == 2 * 32 * 28 * 28 * 240 * 1 * 25
    # strided: 56 -> 28
    assert bench.out_hw(LAYERS["strided_3x3_s2_f32"]) == (28, 28)


def test_bytes_count_every_operand_once():
    L = LAYERS["resnet50_1x1_res_f16"]  # bias and residual, fp16
    x = 32 * 64 * 56 * 56
    w = 256 * 64
    y = 32 * 256 * 56 * 56
    assert bench.layer_bytes(L) == (x + w + 256 + y + y) * 2
    L2 = dataclasses.replace(L, residual_shape=None, bias=False)
    assert bench.layer_bytes(L2) == (x + w + y) * 2


def test_binding_rooflines_of_the_workloads():
    pk = {"hbm_gbs": 6783.8, "bf16_tflops": 1916.3, "bf16_tflops_sustained": 1707.7, "source": "measured"}
    expect = {"resnet50_stem_f16": ("igemm_tcgen05_window", "hbm"),
              "resnet50_3x3_f16": ("igemm_tcgen05_window", "tensor"),
              "resnet50_1x1_res_f16": ("igemm_tcgen05_window", "hbm"),
              "mbv3_pw1x1_f16": ("pointwise_mma", "hbm"),
              "mbv3_dw5x5_f32": ("depthwise_halo", "hbm"),
              "mbv3_pw1x1_f32": ("igemm_ffma", "alu"),
              "strided_3x3_s2_f32": ("igemm_ffma", "alu"),
              "small_3x3_f32": ("igemm_ffma", "hbm")}
    for name, (variant, bound) in expect.items():
        b, peak, unit = bench.roofline_bound(LAYERS[name], variant, pk)
        assert b == bound, (name, b)
        assert unit == ("GB/s" if b == "hbm" else "TFLOP/s")
        assert peak == {"hbm": 6783.8, "tensor": 1916.3, "alu": bench.FFMA_PEAK_TFLOPS}[b]


def test_whole_job_rate_and_single_rank_max():
    assert bench.aggregate(10.0, 4, 2.0) == 20.0  # units of all ranks over the slowest time
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_traffic_only_from_an_unchanged_kernel_source():
    """profiled_traffic returns a summary's DRAM bytes only when the summary's
    source hash is the current source's."""
    for name in os.listdir(os.path.join(bench.ROOT, "profiles")):
        if not name.startswith("igemm_tcw_resnet50_stem_f16"):
            continue
        text = open(os.path.join(bench.ROOT, "profiles", name)).read()
        src = bench.kernel_source("igemm_tcgen05_window")
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        got = bench.profiled_traffic("resnet50_stem_f16", "igemm_tcgen05_window")
        if f"source_sha256_16: {digest}" in text:
            assert got is not None and got > 0
        else:
            assert got is None
