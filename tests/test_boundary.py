"""The C ABI on the host (no GPU needed): the library loads, exports every
symbol include/conv.h declares, validates problems with checked arithmetic,
and plans deterministically.  No compute call is made here."""
import ctypes
import os
import re

import pytest

import implicit_gemm_cnn_gb300 as conv
import oracle
from implicit_gemm_cnn_gb300 import build as conv_build
from workloads import LAYERS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    conv_build.build()
    return conv.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "conv.h")).read()
    return re.findall(r"CONV_API\s+[\w\s\*]+?\b(conv_\w+)\s*\(", text)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) == 18, names
    for name in names:
        assert hasattr(lib, name), name           # dlsym succeeds
    assert conv.conv_abi_version() == 1


def test_struct_layout_matches_header():
    # int64 x 16, then int32, float, float, int32 x 3, uint32 -> 156 -> padded 160
    assert ctypes.sizeof(conv.ConvProblem) == 160
    assert conv.ConvProblem.act.offset == 128 and conv.ConvProblem.flags.offset == 152
    assert ctypes.sizeof(conv.ConvPlanInfo) == 72


def test_status_strings(lib):
    for code in range(11):
        assert conv.conv_status_string(code)


@pytest.mark.parametrize("case", [
    # (x_shape, w_shape, stride, pads, dilation)
    ((1, 1, 4, 4), (1, 1, 3, 3), 1, 0, 1),
    ((8, 3, 224, 224), (64, 3, 7, 7), 2, 3, 1),
    ((1, 1, 10, 10), (1, 1, 3, 3), 1, 0, 2),
    ((2, 4, 13, 9), (6, 4, 4, 2), (3, 2), (2, 0, 1, 3), (1, 3)),
    ((1, 2, 1, 50), (3, 2, 1, 5), 1, (0, 2, 0, 2), 1),      # one-dimensional (h = 1)
    ((1, 2, 5, 5), (2, 2, 5, 5), 1, 0, 1),                    # single output position
])
def test_output_shape_matches_oracle(lib, case):
    xs, ws, stride, pads, dil = case
    p = conv.make_problem(xs, ws, stride=stride, pads=pads, dilation=dil)
    o = oracle.Oracle()
    pt, pl, pb, pr = conv._pads(pads)
    sh, sw = conv._pair(stride)
    dh, dw = conv._pair(dil)
    want = (o.output_extent(xs[2], ws[2], pt, pb, sh, dh), o.output_extent(xs[3], ws[3], pl, pr, sw, dw))
    assert conv.conv_output_shape(p) == want


def _status(fn, *args):
    try:
        fn(*args)
    except conv.ConvError as e:
        return e.name
    return "CONV_OK"


def test_validation_errors(lib):
    ok = dict(x_shape=(2, 4, 8, 8), w_shape=(6, 2, 3, 3), groups=2, pads=1)
    assert _status(conv.conv_output_shape, conv.make_problem(**ok)) == "CONV_OK"
    bad = [
        (dict(ok, x_shape=(0, 4, 8, 8)), "CONV_ERR_SHAPE"),
        (dict(ok, groups=3), "CONV_ERR_SHAPE"),                         # 4 % 3
        (dict(ok, w_shape=(5, 2, 3, 3)), "CONV_ERR_SHAPE"),             # 5 % 2
        (dict(ok, pads=0, w_shape=(6, 2, 9, 9)), "CONV_ERR_SHAPE"),     # no output position
        (dict(ok, pads=(-1, 0, 0, 0)), "CONV_ERR_SHAPE"),
        (dict(ok, stride=0), "CONV_ERR_SHAPE"),
        (dict(ok, dilation=0), "CONV_ERR_SHAPE"),
        (dict(ok, x_shape=(2 ** 40, 4, 2 ** 20, 2 ** 20)), "CONV_ERR_OVERFLOW"),
        (dict(ok, dilation=2 ** 62), "CONV_ERR_OVERFLOW"),
        (dict(ok, x_shape=(1, 4, 70000, 70000)), "CONV_ERR_SHAPE"),     # per-image > int32
    ]
    for kw, want in bad:
        assert _status(conv.conv_output_shape, conv.make_problem(**kw)) == want, (kw, want)
    p = conv.make_problem(**ok)
    p.dtype = 7
    assert _status(conv.conv_output_shape, p) == "CONV_ERR_DTYPE"
    p = conv.make_problem(**ok)
    p.act = 42
    assert _status(conv.conv_output_shape, p) == "CONV_ERR_ACT"
    assert lib.conv_output_shape(None, None, None) == 5  # CONV_ERR_NULL


def test_forward_host_side_errors(lib):
    """Errors conv_forward reports before it touches a device (fake addresses
    are never dereferenced on these paths)."""
    p = conv.make_problem((1, 4, 8, 8), (4, 4, 3, 3), pads=1, has_bias=True)
    x, w, b, y = 0x10000, 0x20000, 0x30000, 0x40000
    assert lib.conv_forward(ctypes.byref(p), None, w, b, None, y, None, 0, None) == 5
    assert lib.conv_forward(ctypes.byref(p), x, w, None, None, y, None, 0, None) == 5  # bias
    # y overlapping the input
    assert lib.conv_forward(ctypes.byref(p), x, w, b, None, x + 64, None, 0, None) == 7
    p.has_residual = 1
    assert lib.conv_forward(ctypes.byref(p), x, w, b, None, y, None, 0, None) == 5
    assert lib.conv_forward(ctypes.byref(p), x, w, b, y, y, None, 0, None) == 7        # in-place
    # no GPU in this process: the device query fails cleanly
    import torch
    if not torch.cuda.is_available():
        p.has_residual = 0
        assert lib.conv_forward(ctypes.byref(p), x, w, b, None, y, None, 0, None) == 8
        assert _status(conv.conv_scratch_bytes, p) == "CONV_ERR_DEVICE"
        assert _status(conv.conv_device_error, True) == "CONV_ERR_DEVICE"


def _layer_problem(L, flags=0):
    return conv.make_problem((L.n, L.c_in, L.h, L.w), (L.c_out, L.c_in // L.groups, L.kh, L.kw),
                             dtype=L.dtype, stride=L.stride, pads=L.pads, dilation=L.dilation,
                             groups=L.groups, act=L.act, alpha=L.alpha, has_bias=L.bias,
                             has_residual=L.residual_shape is not None, flags=flags)


EXPECTED_VARIANT = {
    "small_3x3_f32": "igemm_ffma", "resnet50_stem_f16": "igemm_tcgen05_window",
    "resnet50_3x3_f16": "igemm_tcgen05_window", "resnet50_1x1_res_f16": "igemm_tcgen05_window",
    "mbv3_dw5x5_f32": "depthwise_halo", "mbv3_dw5x5_f16": "depthwise_halo",
    "mbv3_pw1x1_f32": "igemm_ffma", "mbv3_pw1x1_f16": "pointwise_mma",
    "grouped_dil2_f32": "igemm_ffma", "late_1x1_splitk_f32": "igemm_ffma_split_k",
    "strided_3x3_s2_f32": "igemm_ffma",
    "resnet50_3x3_256_f32": "winograd_f2x2_3x3",
}


UNFOLDED = {"strided_3x3_s2_f32"}   # CUDA-core layers planned with the unfolded-input pre-pass


@pytest.mark.parametrize("name", sorted(LAYERS))
def test_plans_of_the_workloads(lib, name):
    L = LAYERS[name]
    p = _layer_problem(L)
    plan = conv.conv_plan(p, 152)
    assert plan["variant_name"] == EXPECTED_VARIANT[name], plan
    assert (plan["ho"], plan["wo"]) == conv.conv_output_shape(p)
    assert plan["gemm_k"] == (L.c_in // L.groups) * L.kh * L.kw
    assert plan["gemm_n"] == L.n * plan["ho"] * plan["wo"]
    y_elems = L.n * L.c_out * plan["ho"] * plan["wo"]
    if plan["split_k"] > 1:
        assert plan["scratch_bytes"] == plan["split_k"] * y_elems * 4
        assert plan["ctas"] <= 2 * 152
    elif plan["variant_name"] == "igemm_tcgen05_window":
        tile = plan["tile_m"]
        assert tile % 16 == 0 and tile <= 256
        # repacked weights: channel tiles x k blocks x tile channels x 16 bytes
        assert plan["scratch_bytes"] % (16 * tile) == 0
        assert plan["scratch_bytes"] >= L.c_out * (L.c_in // L.groups) * L.kh * L.kw * 2
        assert plan["ctas"] <= 152
        p2 = _layer_problem(L, flags=conv.FLAG_NO_WINDOW)
        assert conv.conv_plan(p2, 152)["variant_name"] == "igemm_tcgen05"
        assert conv.conv_plan(p2, 152)["scratch_bytes"] == 0
    elif plan["variant_name"] == "pointwise_mma":
        # one block per 128-pixel block of an image and channel block, no scratch
        assert plan["scratch_bytes"] == 0 and plan["tile_n"] == 128
        bm = plan["tile_m"]
        assert L.c_out <= 64 and bm == (L.c_out + 15) // 16 * 16
        hw = plan["ho"] * plan["wo"]
        assert plan["ctas"] == L.n * -(-hw // 128) * -(-L.c_out // bm)
        # with the kernel turned off: the shifted-window kernel's 1x1 view
        p2 = _layer_problem(L, flags=conv.FLAG_NO_PW_MMA)
        assert conv.conv_plan(p2, 152)["variant_name"] == "igemm_tcgen05_window"
    elif name in UNFOLDED:
        # the unfolded input (float32 n x c_in x kw x hu x Wo, hu the padded
        # rows the windows reach) on a 256-byte boundary, then the transposed
        # weights (groups x k x channels rounded to 4)
        hu = (plan["ho"] - 1) * L.stride[0] + (L.kh - 1) * L.dilation[0] + 1
        xw = L.n * L.c_in * L.kw * hu * plan["wo"] * 4
        mg4 = (L.c_out // L.groups + 3) // 4 * 4
        wt = L.groups * plan["gemm_k"] * mg4 * 4
        base = (xw + 255) // 256 * 256 + wt
        # a tail split: the tiles of the last, partly filled round (2 blocks of
        # 128 x 128 per SM) run as s k ranges each, their raw tiles after the
        # weights
        tiles = -(-plan["gemm_n"] // plan["tile_n"]) * -(-plan["gemm_m"] // plan["tile_m"])
        if plan["ctas"] > tiles:
            rest = tiles % (2 * 152)
            s_ranges = 1 + (plan["ctas"] - tiles) // rest
            assert plan["ctas"] == tiles - rest + rest * s_ranges and 2 <= s_ranges <= 8
            base = (base + 255) // 256 * 256 + rest * s_ranges * plan["tile_m"] * plan["tile_n"] * 4
        assert plan["scratch_bytes"] == base
        p2 = _layer_problem(L, flags=conv.FLAG_NO_UNFOLD)
        assert conv.conv_plan(p2, 152)["scratch_bytes"] == 0
    elif plan["variant_name"] == "winograd_f2x2_3x3":
        # U[16][K][C], V[16][C][tiles rounded to 4], M[16][K][same], 256-byte aligned
        tiles = L.n * -(-plan["ho"] // 2) * -(-plan["wo"] // 2)
        p4 = (tiles + 3) // 4 * 4
        u = (16 * L.c_out * L.c_in * 4 + 255) // 256 * 256
        v = (16 * L.c_in * p4 * 4 + 255) // 256 * 256
        assert plan["scratch_bytes"] == u + v + 16 * L.c_out * p4 * 4
    else:
        assert plan["scratch_bytes"] == 0
    assert conv.conv_plan(p, 152) == plan      # a pure function of (problem, SMs)


def test_split_k_rule(lib):
    L = LAYERS["late_1x1_splitk_f32"]
    p = _layer_problem(L)
    a, b = conv.conv_plan(p, 152), conv.conv_plan(p, 148)
    assert a["split_k"] > 1 and b["split_k"] > 1
    # at most 16 ranges of at least 128 terms each (whole pipeline stages), covering k
    K = a["gemm_k"]
    per = -(-K // a["split_k"])
    assert a["split_k"] <= 16 and K / a["split_k"] >= 128
    # forcing: none, or an exact count
    q = _layer_problem(L, flags=conv.FLAG_NO_SPLIT_K)
    assert conv.conv_plan(q, 152)["split_k"] == 1 and conv.conv_plan(q, 152)["scratch_bytes"] == 0
    q = _layer_problem(L, flags=4 << conv.SPLIT_K_SHIFT)
    assert conv.conv_plan(q, 152)["split_k"] == 4
    # a grid that already fills the device does not split
    big = LAYERS["strided_3x3_s2_f32"]
    assert conv.conv_plan(_layer_problem(big), 152)["split_k"] == 1
    assert per >= 128


def test_force_ffma_flag(lib):
    for name in ("resnet50_stem_f16", "mbv3_dw5x5_f32"):
        p = _layer_problem(LAYERS[name], flags=conv.FLAG_FORCE_FFMA)
        assert conv.conv_plan(p, 152)["variant_name"].startswith("igemm_ffma")


def test_plan_rejects_bad_sm_count(lib):
    p = _layer_problem(LAYERS["small_3x3_f32"])
    assert _status(conv.conv_plan, p, 0) == "CONV_ERR_ARG"


def test_grouped_layers_take_the_staged_rows_path(lib):
    """fp32 grouped layers with Cout/groups a multiple of 8 (at most 64), stride
    1, a square 3x3 or 5x5 kernel and Wo a multiple of 4 run the grouped path:
    tile = the group's output channels x 8 output rows, no scratch, no split."""
    p = conv.make_problem((16, 512, 28, 28), (512, 16, 3, 3), dtype="f32", pads=2, dilation=2, groups=32,
                          act="silu", has_bias=True)
    plan = conv.conv_plan(p, 152)
    assert plan["variant_name"] == "igemm_ffma" and plan["split_k"] == 1 and plan["scratch_bytes"] == 0
    assert (plan["tile_m"], plan["tile_n"]) == (16, 8 * 28)
    # outside the path: Cout/groups of 4, stride 2, Wo of 15, fp16
    for xs, ws, g, dt in [((2, 16, 12, 12), (8, 8, 3, 3), dict(pads=1, groups=2), "f32"),
                          ((2, 16, 12, 12), (16, 8, 3, 3), dict(pads=1, groups=2, stride=2), "f32"),
                          ((2, 16, 12, 15), (16, 8, 3, 3), dict(pads=1, groups=2), "f32")]:
        q = conv.conv_plan(conv.make_problem(xs, ws, dtype=dt, **g), 152)
        assert q["tile_n"] != 8 * conv.conv_output_shape(conv.make_problem(xs, ws, dtype=dt, **g))[1], q



def test_planner_rules_on_random_shapes(lib):
    """Seeded random problems: every valid one plans, deterministically, and
    the variant respects what each kernel takes -- depthwise for one input
    channel per group, the shifted-window kernel only for 16-bit, one group,
    stride 1 or 2 (dilation 1) and rows of 8-element multiples,
    tensor-core variants never for fp32, split k only with its planes in
    scratch."""
    import random
    rng = random.Random(20260101)
    seen = set()
    for _ in range(300):
        dt = rng.choice(["f32", "f16", "bf16"])
        groups = rng.choice([1, 1, 1, 2, 4, 8])
        cg = rng.choice([1, 3, 4, 8, 16, 24, 64])
        mg = rng.choice([1, 2, 8, 16, 40])
        k = rng.choice([1, 3, 5, 7])
        kh, kw = (k, k) if rng.random() < 0.8 else (k, rng.choice([1, 3]))
        s = rng.choice([1, 1, 2, 3])
        d = rng.choice([1, 1, 2])
        n, h, w = rng.choice([1, 2, 4]), rng.randint(kh, 40), rng.randint(kw, 48)
        pads = tuple(rng.randint(0, 3) for _ in range(4))
        p = conv.make_problem((n, cg * groups, h, w), (mg * groups, cg, kh, kw), dtype=dt, stride=s, pads=pads,
                              dilation=d, groups=groups, has_bias=rng.random() < 0.5,
                              has_residual=rng.random() < 0.3)
        try:
            ho, wo = conv.conv_output_shape(p)
        except conv.ConvError:
            continue  # the kernel does not fit the padded input
        plan = conv.conv_plan(p, 152)
        assert conv.conv_plan(p, 152) == plan
        v = plan["variant_name"]
        seen.add(v)
        assert (plan["ho"], plan["wo"]) == (ho, wo)
        if cg == 1:
            assert v == "depthwise_halo", (p, plan)
        if dt == "f32":
            assert v in ("igemm_ffma", "igemm_ffma_split_k", "depthwise_halo"), (p, plan)
        if v == "pointwise_mma":
            assert dt != "f32" and kh == kw == 1 and s == 1 and not any(pads) and groups == 1 and mg <= 64, (p, plan)
            assert plan["scratch_bytes"] == 0
        if v == "igemm_tcgen05_window":
            # rows of 8-element multiples: the output's, or for a 1x1 layer
            # read as it lies, a row length dividing the plane
            pointwise = kh == kw == 1 and s == 1 and not any(pads)
            assert dt != "f32" and groups == 1, (p, plan)
            assert wo % 8 == 0 or (pointwise and (ho * wo) % 8 == 0), (p, plan)
            assert s == 1 or (s == 2 and d == 1), (p, plan)
            assert plan["scratch_bytes"] > 0 and plan["scratch_bytes"] % 16 == 0
        if v == "igemm_ffma_split_k":
            assert plan["split_k"] > 1 and plan["scratch_bytes"] == plan["split_k"] * n * mg * groups * ho * wo * 4
        else:
            assert plan["split_k"] == 1
    assert {"igemm_ffma", "depthwise_halo", "pointwise_mma", "igemm_tcgen05"} <= seen, seen


# ---- ONNX auto_pad ----------------------------------------------------------
AUTO_PAD_HAND = [
    # (size, k, stride, dilation) -> SAME_UPPER (begin, end), SAME_LOWER (begin, end);
    # worked by hand: out = ceil(size / stride), total = (out-1)*s + d(k-1) + 1 - size
    ((224, 7, 2, 1), (2, 3), (3, 2)),     # out 112, total 5 (the ResNet-50 stem)
    ((56, 3, 1, 1), (1, 1), (1, 1)),      # out 56, total 2
    ((5, 2, 1, 1), (0, 1), (1, 0)),       # out 5, total 1
    ((7, 3, 2, 2), (2, 2), (2, 2)),       # out 4, total 4
    ((8, 1, 2, 1), (0, 0), (0, 0)),       # out 4, total max(0, -1) = 0
    ((10, 4, 3, 1), (1, 2), (2, 1)),      # out 4, total 3
]


@pytest.mark.parametrize("case", AUTO_PAD_HAND)
def test_auto_pad_oracle_hand_values(case):
    """The oracle's auto_pad against values worked by hand from ONNX's rule."""
    from oracle import arith
    (size, k, s, d), upper, lower = case
    assert arith.auto_pad(size, k, s, d, "SAME_UPPER") == upper
    assert arith.auto_pad(size, k, s, d, "SAME_LOWER") == lower
    assert arith.auto_pad(size, k, s, d, "VALID") == (0, 0)


def test_auto_pad_oracle_same_output_size():
    """SAME padding's defining property: the output has ceil(size / stride)
    positions (ONNX), and the two sides differ by at most one."""
    from oracle import arith
    o = oracle.Oracle()
    for size in range(1, 30):
        for k in (1, 2, 3, 5, 7):
            for s in (1, 2, 3):
                for d in (1, 2):
                    for mode in ("SAME_UPPER", "SAME_LOWER"):
                        b, e = arith.auto_pad(size, k, s, d, mode)
                        assert abs(b - e) <= 1 and b >= 0 and e >= 0
                        assert (b <= e) == (mode == "SAME_UPPER" or b == e)
                        if size + b + e >= d * (k - 1) + 1:
                            assert o.output_extent(size, k, b, e, s, d) == -(-size // s), (size, k, s, d)


def test_auto_pad_c_abi_matches_oracle(lib):
    from oracle import arith
    for (h, w) in ((224, 224), (13, 9), (5, 40), (1, 17)):
        for (kh, kw) in ((7, 7), (3, 2), (1, 5)):
            for (sh, sw) in ((1, 1), (2, 2), (3, 1)):
                for (dh, dw) in ((1, 1), (2, 1)):
                    for mode in ("SAME_UPPER", "SAME_LOWER", "VALID"):
                        p = conv.make_problem((2, 3, h, w), (4, 3, kh, kw), stride=(sh, sw),
                                              dilation=(dh, dw), pads=(9, 9, 9, 9))
                        if mode == "VALID" and (h < (kh - 1) * dh + 1 or w < (kw - 1) * dw + 1):
                            st = lib.conv_apply_auto_pad(ctypes.byref(p), conv.AUTO_PAD[mode])
                            assert conv.STATUS[st] == "CONV_ERR_SHAPE"
                            assert (p.pad_top, p.pad_left) == (9, 9)    # unchanged on error
                            continue
                        conv.conv_apply_auto_pad(p, mode)
                        pt, pb = arith.auto_pad(h, kh, sh, dh, mode)
                        pl, pr = arith.auto_pad(w, kw, sw, dw, mode)
                        assert (p.pad_top, p.pad_left, p.pad_bottom, p.pad_right) == (pt, pl, pb, pr)
                        if mode != "VALID":
                            assert conv.conv_output_shape(p) == (-(-h // sh), -(-w // sw))
    p = conv.make_problem((1, 1, 8, 8), (1, 1, 3, 3), pads=(1, 2, 3, 4))
    conv.conv_apply_auto_pad(p, "NOTSET")
    assert (p.pad_top, p.pad_left, p.pad_bottom, p.pad_right) == (1, 2, 3, 4)
    assert conv.STATUS[lib.conv_apply_auto_pad(ctypes.byref(p), 7)] == "CONV_ERR_ARG"
    assert conv.STATUS[lib.conv_apply_auto_pad(None, 1)] == "CONV_ERR_NULL"


# ---- the description of a plan, on the host -----------------------------------
def test_describe_plan_matches_plan(lib):
    """conv_describe_plan (host only) names the planned variant, its blocks,
    split and scratch as conv_plan reports them, and ends with the launch count."""
    for name, L in LAYERS.items():
        if name not in EXPECTED_VARIANT:
            continue
        p = _layer_problem(L)
        plan = conv.conv_plan(p, 152)
        desc = conv.conv_describe_plan(p, 152)
        assert desc.split()[0] == plan["variant_name"] == EXPECTED_VARIANT[name], (name, desc)
        assert desc.endswith(" launches=%d" % int(re.search(r"launches=(\d+)$", desc).group(1)))
        assert "sms=152" in desc, desc
        if plan["variant_name"].startswith("igemm_ffma") and "grouped" not in desc:
            assert "split_k=%d" % plan["split_k"] in desc and "blocks=%d" % plan["ctas"] in desc, desc
            assert "scratch=%d" % plan["scratch_bytes"] in desc, desc
        assert conv.conv_describe_plan(p, 152) == desc      # a pure function of (problem, SMs)


def test_describe_plan_launch_counts(lib):
    """Kernels one call launches, per variant: the shifted-window kernel and its
    weight repack 2, Winograd's transforms and products 4, the unfolded CUDA-core
    path (pre-pass, kernel, tail reduction) 3, a single kernel otherwise."""
    want = {"resnet50_stem_f16": 2, "resnet50_3x3_f16": 2, "resnet50_1x1_res_f16": 2,
            "mbv3_dw5x5_f32": 1, "mbv3_dw5x5_f16": 1, "mbv3_pw1x1_f16": 1, "mbv3_pw1x1_f32": 1,
            "grouped_dil2_f32": 1, "small_3x3_f32": 1, "strided_3x3_s2_f32": 3,
            "resnet50_3x3_256_f32": 4}
    for name, n in want.items():
        desc = conv.conv_describe_plan(_layer_problem(LAYERS[name]), 152)
        assert desc.endswith("launches=%d" % n), (name, desc)


def test_describe_plan_split_k_reduction(lib):
    """Split k: the ranges of a tile reduced within a thread-block cluster (one
    launch) up to 16 ranges; the float32 planes and a second kernel under
    CONV_FLAG_NO_CLUSTER_K or past 16 ranges."""
    L = LAYERS["late_1x1_splitk_f32"]
    desc = conv.conv_describe_plan(_layer_problem(L), 152)
    assert "split_k=16 reduce=cluster" in desc and desc.endswith("launches=1"), desc
    desc = conv.conv_describe_plan(_layer_problem(L, flags=conv.FLAG_NO_CLUSTER_K), 152)
    assert "split_k=16 reduce=planes" in desc and desc.endswith("launches=2"), desc
    desc = conv.conv_describe_plan(_layer_problem(L, flags=32 << conv.SPLIT_K_SHIFT), 152)
    assert "split_k=32 reduce=planes" in desc and desc.endswith("launches=2"), desc
    desc = conv.conv_describe_plan(_layer_problem(L, flags=conv.FLAG_NO_SPLIT_K), 152)
    assert "split_k=1 " in desc and "reduce=" not in desc and desc.endswith("launches=1"), desc
    # the plan (and so the scratch figure) does not depend on the reduction's form
    a = conv.conv_plan(_layer_problem(L), 152)
    b = conv.conv_plan(_layer_problem(L, flags=conv.FLAG_NO_CLUSTER_K), 152)
    assert a == b


def test_describe_plan_errors(lib):
    p = _layer_problem(LAYERS["small_3x3_f32"])
    buf = ctypes.create_string_buffer(64)
    assert lib.conv_describe_plan(ctypes.byref(p), 0, buf, len(buf)) == 10           # CONV_ERR_ARG
    assert lib.conv_describe_plan(ctypes.byref(p), 152, None, 0) == 5               # CONV_ERR_NULL
    short = ctypes.create_string_buffer(8)
    assert lib.conv_describe_plan(ctypes.byref(p), 152, short, len(short)) == 0     # truncated, terminated
    assert len(short.value) == 7
    bad = conv.make_problem((1, 3, 2, 2), (16, 3, 3, 3))                            # no output position
    with pytest.raises(conv.ConvError):
        conv.conv_describe_plan(bad, 152)
