"""Benchmark of the forward convolution on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--layer NAME | --layers all]

One step is one conv_forward over one batch of the workload layer: by
default the largest configuration by arithmetic, N=16 256->512 3x3 stride 2
pad 1 on 56x56 with leaky-relu 0.1 in fp32 (14.8 G multiply-adds).  Inputs are seeded synthetic tensors of the layer's shapes
and distributions, resident in HBM; the step rotates over enough independent
input sets that their total exceeds twice the L2, so every step reads its
operands from HBM.  The K timed steps are replayed from CUDA graphs of
back-to-back launches; the region is bracketed by a barrier and device
synchronisation, timed with CUDA events, and the max over ranks is taken.

The JSON line also carries: the roofline of one call (algorithmic bytes or
FLOPs of one call over its average duration in the timed region, measured with
the CUDA events around that region, against the measured peaks), the end-to-end rate
through the public API with pinned host buffers, the CPU oracle's rate on a
bounded sample (test infrastructure, timed only here), the kernel launch
count and the SM clocks seen.

The default run also times every other workload layer (fewer steps, no
end-to-end or CPU legs) and nests their rates -- TFLOP/s for every layer and
GB/s for the depthwise ones -- under "layers" in the same single JSON line.

--impl reference times the CPU oracle itself on the same workload and metric,
one bounded sample per step.  --layers all prints one full line per workload
layer.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "conv TFLOP/s (2·N·Ho·Wo·Co·Ci·k²/g) and depthwise GB/s, % of roofline"
HEADLINE = "strided_3x3_s2_f32"
L2_BYTES = 129 * 1024 * 1024
# float32 FFMA peak: 152 SMs x 128 FMA lanes x 2 FLOP x 2.07 GHz (maximum SM clock)
FFMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


# ---- layer arithmetic (closed forms; no convolution is evaluated here) -----
def out_hw(L):
    ho = (L.h + L.pads[0] + L.pads[2] - L.dilation[0] * (L.kh - 1) - 1) // L.stride[0] + 1
    wo = (L.w + L.pads[1] + L.pads[3] - L.dilation[1] * (L.kw - 1) - 1) // L.stride[1] + 1
    return ho, wo


def layer_flops(L) -> int:
    ho, wo = out_hw(L)
    return 2 * L.n * ho * wo * L.c_out * (L.c_in // L.groups) * L.kh * L.kw


def layer_bytes(L) -> int:
    """Algorithmic bytes: every operand read once, the output written once."""
    ho, wo = out_hw(L)
    es = 4 if L.dtype == "f32" else 2
    y = L.n * L.c_out * ho * wo
    elems = (L.n * L.c_in * L.h * L.w + L.c_out * (L.c_in // L.groups) * L.kh * L.kw
             + (L.c_out if L.bias else 0) + (y if L.residual_shape else 0) + y)
    return elems * es


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def roofline_bound(L, variant: str, pk: dict) -> tuple[str, float, str]:
    """(bound, peak, unit) of the layer's binding roofline: HBM when its
    arithmetic intensity is below the ridge of its compute path."""
    intensity = layer_flops(L) / layer_bytes(L)
    if variant.startswith("depthwise"):
        # a direct stencil doing k*k multiply-adds per value it reads: its
        # roofline is HBM ("Convolutions", 2.3: the depthwise layer's low
        # arithmetic intensity)
        return "hbm", pk["hbm_gbs"], "GB/s"
    if variant.startswith("igemm_tcgen05"):
        compute, kind = pk["bf16_tflops"], "tensor"  # fp16 and bf16 share the dense rate
    elif variant.startswith("pointwise_mma"):
        compute, kind = MMA_SYNC_PEAK_TFLOPS, "tensor"  # the warp-level MMA path's own rate
    else:
        compute, kind = FFMA_PEAK_TFLOPS, "alu"
    ridge = compute * 1e12 / (pk["hbm_gbs"] * 1e9)
    if intensity < ridge:
        return "hbm", pk["hbm_gbs"], "GB/s"
    return kind, compute, "TFLOP/s"


def kernel_source(variant: str) -> str:
    name = {"igemm_tcgen05": "conv_tc.cu", "igemm_tcgen05_window": "conv_tcw.cu",
            "depthwise_halo": "conv_depthwise.cu", "pointwise_mma": "conv_pointwise.cu"}.get(variant.split()[0],
                                                                                             "conv_ffma.cu")
    return os.path.join(ROOT, "implicit_gemm_cnn_gb300", "csrc", name)


def profiled_traffic(layer_name: str, variant: str, source: str | None = None):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if the kernel source is unchanged since the capture (`source`:
    the dominant kernel's file under csrc/, else the variant's)."""
    src = (os.path.join(ROOT, "implicit_gemm_cnn_gb300", "csrc", source) if source else kernel_source(variant))
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    prof_dir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof_dir):
        return None
    for fn in sorted(os.listdir(prof_dir)):
        if layer_name not in fn:
            continue
        text = open(os.path.join(prof_dir, fn)).read()
        m = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
        t = re.search(r"dram_bytes_per_launch:\s*([0-9.e+]+)", text)
        if m and t and m.group(1) == digest:
            return float(t.group(1))
    return None


# ---- distributed helpers (also exercised by the CPU gloo tests) ----------
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(per_rank_units: float, world: int, seconds_max: float) -> float:
    """Whole-job rate: units of all ranks over the slowest rank's time."""
    return per_rank_units * world / seconds_max


# ---- clocks --------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---- our implementation --------------------------------------------------
def run_ours(L, steps: int, warmup: int, world: int, rank: int, local_rank: int,
             with_cpu_baseline: bool, with_e2e: bool, quick: bool = False) -> dict:
    import torch

    import implicit_gemm_cnn_gb300 as conv
    from workloads import make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    geo = dict(stride=L.stride, pads=L.pads, dilation=L.dilation, groups=L.groups, act=L.act,
               alpha=L.alpha, beta=L.beta)
    p = conv.make_problem((L.n, L.c_in, L.h, L.w), (L.c_out, L.c_in // L.groups, L.kh, L.kw),
                          dtype=L.dtype, has_bias=L.bias, has_residual=L.residual_shape is not None,
                          **geo)
    ho, wo = conv.conv_output_shape(p)
    variant = conv.conv_describe_variant(p)
    need = conv.conv_scratch_bytes(p)
    plan = conv.conv_plan(p, torch.cuda.get_device_properties(local_rank).multi_processor_count)
    # kernels one call launches, as the library describes its plan
    m = re.search(r"launches=(\d+)", variant)
    if not m:
        raise RuntimeError(f"variant description without a launch count: {variant}")
    launches_per_step = int(m.group(1))
    set_bytes = layer_bytes(L)
    nsets = max(1, min(256, math.ceil(2 * L2_BYTES / set_bytes)))  # tiny layers stay L2-resident
    sets = []
    for s in range(nsets):
        inp = make_inputs(L, seed_offset=s + 1000 * rank)
        t = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
        t["y"] = torch.empty((L.n, L.c_out, ho, wo), dtype=t["x"].dtype, device=dev)
        t["scratch"] = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        sets.append(t)

    def step(i):
        t = sets[i % nsets]
        conv.conv_forward(p, t["x"], t["w"], t["bias"], t["residual"], t["y"], t["scratch"], need)

    # W untimed warm-up steps through the public call
    for i in range(max(warmup, nsets)):
        step(i)
    torch.cuda.synchronize()

    # graphs of back-to-back calls (no event nodes between the steps: they
    # would add their own gaps to the timed region)
    chunk = max(1, min(steps, max(nsets, 500)))

    def capture(n):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                step(i)
        torch.cuda.synchronize()
        return g

    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if quick:
        # eager launches, no graphs or clock settling: for profiler captures
        sampler = ClockSampler(local_rank).start()
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        clocks = sampler.stop()
    else:
        g_full = capture(chunk)
        full_reps, rem = divmod(steps, chunk)
        g_rem = capture(rem) if rem else None
        # settle clocks under load (untimed); clocks are sampled through the timed region
        sampler = ClockSampler(local_rank).start()
        t_end = time.time() + 1.0
        while time.time() < t_end:
            g_full.replay()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(full_reps):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        clocks = sampler.stop()
    secs = e0.elapsed_time(e1) / 1e3
    secs_max = max_over_ranks(secs, world)

    # average duration of one call (all its kernels, back to back in the
    # graphs), from the CUDA events around the timed region
    launch_ms = secs * 1e3 / steps

    flops = layer_flops(L)
    value = aggregate(flops * steps, world, secs_max) / 1e12
    pk = peaks()
    bound, peak, unit = roofline_bound(L, variant, pk)
    per_launch = layer_bytes(L) if bound == "hbm" else flops
    achieved = per_launch / (launch_ms / 1e3) / (1e9 if unit == "GB/s" else 1e12)
    roof = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": profiled_traffic(L.name, variant),
            "peak_source": pk["source"], "algorithmic_per_launch": per_launch,
            "launch_us": round(launch_ms * 1e3, 3),
            "tensor_or_alu_frac": round(flops / (launch_ms / 1e3) / 1e12 / (
                pk["bf16_tflops"] if variant.startswith("igemm_tcgen05") else FFMA_PEAK_TFLOPS), 4)}

    out = {"value": value, "secs": secs_max, "variant": variant, "roofline": roof,
           "clocks": clocks, "launches": launches_per_step * steps, "nsets": nsets,
           "set_bytes": set_bytes, "chunk": chunk}

    if with_e2e:
        out["e2e"] = e2e_rate(L, p, sets[0], need, min(steps, 200), dev)
    if with_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(L, target_s=10.0)
    return out


def e2e_rate(L, p, t, need, steps, dev) -> dict:
    """Through the public API, every step: the step's x from pinned host memory
    to the device, the convolution, its y back to pinned host memory.  The
    library's HostPipeline overlaps one step's copies with its neighbours'
    convolutions (three streams, two device buffers each of x and y)."""
    import torch

    import implicit_gemm_cnn_gb300 as conv
    x_host = t["x"].cpu().pin_memory()
    y_hosts = [torch.empty(t["y"].shape, dtype=t["y"].dtype).pin_memory() for _ in range(2)]
    geo = dict(stride=L.stride, pads=L.pads, dilation=L.dilation, groups=L.groups, act=L.act,
               alpha=L.alpha, beta=L.beta)
    pipe = conv.HostPipeline(tuple(t["x"].shape), t["w"], t["bias"], t["residual"], **geo)

    def run(n):
        pipe.run([x_host] * n, [y_hosts[i % 2] for i in range(n)])

    run(4)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    run(steps)
    e1.record(s)
    torch.cuda.synchronize()
    secs = e0.elapsed_time(e1) / 1e3
    return {"value": layer_flops(L) * steps / secs / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
            "d2h_bytes_per_step": y_hosts[0].numel() * y_hosts[0].element_size(), "steps": steps,
            "overlap": "HostPipeline: copies of one step overlap the neighbouring steps' convolutions"}


# ---- the CPU oracle (reported baseline / reference arm) -------------------
def _oracle_setup(L):
    import numpy as np

    import oracle
    from workloads import make_inputs, to_numpy_operand
    inp = make_inputs(L)
    ops = [to_numpy_operand(inp[k], L.dtype) for k in ("x", "w", "bias", "residual")]
    o = oracle.Oracle()
    kw = dict(dtype=L.dtype, stride=L.stride, pads=L.pads, dilation=L.dilation, groups=L.groups,
              act=L.act, alpha=L.alpha, beta=L.beta)
    ho, wo = out_hw(L)
    total = L.n * L.c_out * ho * wo
    per_out_flops = 2 * (L.c_in // L.groups) * L.kh * L.kw
    return o, ops, kw, total, per_out_flops, np


def cpu_baseline(L, target_s: float = 10.0) -> dict:
    """The oracle as it stands on this host's cores, on a bounded sample of
    the workload's outputs (about target_s seconds of CPU work)."""
    o, ops, kw, total, per_out, np = _oracle_setup(L)
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(total, min(total, 20000), replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    o.conv2d(*ops, index=probe, nthreads=cores, **kw)
    rate = len(probe) / max(time.perf_counter() - t0, 1e-6)   # outputs / s
    count = int(min(total, max(len(probe), rate * target_s)))
    idx = np.sort(rng.choice(total, count, replace=False)).astype(np.int64) if count < total else None
    t0 = time.perf_counter()
    o.conv2d(*ops, index=idx, nthreads=cores, **kw)
    secs = time.perf_counter() - t0
    return {"value": count * per_out / secs / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "seconds": round(secs, 2),
            "sample": f"{count} of {total} outputs ({'all' if idx is None else 'random'}) of one "
                      f"batch, float64 sums, {cores} threads"}


def run_reference(L, steps: int, warmup: int) -> dict:
    """The reference arm: the CPU oracle, each step a bounded sample of the
    workload, sized so that the whole run takes about a minute."""
    o, ops, kw, total, per_out, np = _oracle_setup(L)
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(1)
    probe = np.sort(rng.choice(total, min(total, 20000), replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    o.conv2d(*ops, index=probe, nthreads=cores, **kw)
    rate = len(probe) / max(time.perf_counter() - t0, 1e-6)
    per_step = int(max(1, min(total, rate * 60.0 / max(steps + warmup, 1))))
    samples = [np.sort(rng.choice(total, per_step, replace=False)).astype(np.int64)
               for _ in range(min(steps, 64))]
    for i in range(warmup):
        o.conv2d(*ops, index=samples[i % len(samples)], nthreads=cores, **kw)
    t0 = time.perf_counter()
    for i in range(steps):
        o.conv2d(*ops, index=samples[i % len(samples)], nthreads=cores, **kw)
    secs = time.perf_counter() - t0
    value = per_step * per_out * steps / secs / 1e12
    return {"value": value, "secs": secs, "per_step": per_step, "cores": cores, "total": total}


# ---- ConvInteger ---------------------------------------------------------------
# dp4a (4 multiply-adds of bytes into an int32) issues on 64 lanes per SM per
# clock on GB300 -- half the FP32 FFMA rate, measured at 20.0 G instructions/s
# against 39.0 G for FFMA -- so 152 SMs x 64 x 8 ops x 2.07 GHz
DP4A_PEAK_TOPS = 152 * 64 * 4 * 2 * 2.07e9 / 1e12
# Warp-level mma.sync m16n8k16 (f16 in, f32 accumulate) on this GPU: 147.8 G
# MMAs/s x 8192 FLOP = 1210 TFLOP/s, measured by a probe of independent MMA
# chains on every SM (the rate of the kernels that use it, below tcgen05's).
MMA_SYNC_PEAK_TFLOPS = 1210.0


def int_layer_ops(L) -> int:
    ho = (L.h + L.pads[0] + L.pads[2] - L.dilation[0] * (L.kh - 1) - 1) // L.stride[0] + 1
    wo = (L.w + L.pads[1] + L.pads[3] - L.dilation[1] * (L.kw - 1) - 1) // L.stride[1] + 1
    return 2 * L.n * ho * wo * L.c_out * (L.c_in // L.groups) * L.kh * L.kw


def run_integer(L, steps: int, warmup: int, world: int, local_rank: int) -> dict:
    """conv_integer_forward timed like run_ours: CUDA graphs of back-to-back
    calls over input sets rotated past L2, events on the launching stream."""
    import torch

    import implicit_gemm_cnn_gb300 as conv
    from workloads import make_int_inputs
    dev = torch.device("cuda", local_rank)
    geo = dict(stride=L.stride, pads=L.pads, dilation=L.dilation, groups=L.groups)
    p = conv.make_problem((L.n, L.c_in, L.h, L.w), (L.c_out, L.c_in // L.groups, L.kh, L.kw), **geo)
    ho, wo = conv.conv_output_shape(p)
    need = conv.conv_integer_scratch_bytes(p, L.x_type, L.w_type)
    set_bytes = L.n * L.c_in * L.h * L.w + L.c_out * (L.c_in // L.groups) * L.kh * L.kw + 4 * L.n * L.c_out * ho * wo
    nsets = max(1, min(64, math.ceil(2 * L2_BYTES / set_bytes)))
    sets = []
    for i in range(nsets):
        t = {k: v.to(dev) for k, v in make_int_inputs(L, seed_offset=i + 1).items()}
        t["y"] = torch.empty((L.n, L.c_out, ho, wo), dtype=torch.int32, device=dev)
        sets.append(t)
    scratch = torch.empty(need, dtype=torch.uint8, device=dev)

    def step(i):
        t = sets[i % nsets]
        conv.conv_integer_forward(p, L.x_type, L.w_type, t["x"], t["w"], t["x_zero"], t["w_zero"],
                                  t["w_zero"].numel(), t["y"], scratch, need)

    for i in range(max(warmup, nsets)):
        step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for i in range(steps):
            step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank).start()
    t_end = time.time() + 0.5
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    us = secs * 1e6 / steps
    ops = int_layer_ops(L)
    value = aggregate(ops * steps, world, secs) / 1e12
    return {"value": value, "us": us, "clocks": clocks, "launches": 3 * steps,
            "roofline": {"bound": "alu", "achieved": round(ops / (us / 1e6) / 1e12, 2), "peak": DP4A_PEAK_TOPS,
                         "unit": "TOP/s", "frac": round(ops / (us / 1e6) / 1e12 / DP4A_PEAK_TOPS, 4),
                         "traffic": profiled_traffic(L.name, "", "conv_integer.cu"),
                         "tensor_or_alu_frac": round(ops / (us / 1e6) / 1e12 / DP4A_PEAK_TOPS, 4)}}


# ---- ConvTranspose ---------------------------------------------------------------
def transpose_flops(L) -> int:
    """2 x the multiply-adds of the transposed convolution: every input pixel
    times its kernel taps times the output channels of its group."""
    return 2 * L.n * L.c_in * L.h * L.w * (L.c_out // L.groups) * L.kh * L.kw


def run_transpose(L, steps: int, warmup: int, world: int, local_rank: int) -> dict:
    import torch

    import implicit_gemm_cnn_gb300 as conv
    from workloads import make_transpose_inputs
    dev = torch.device("cuda", local_rank)
    p = conv.make_transpose_problem((L.n, L.c_in, L.h, L.w), (L.c_in, L.c_out // L.groups, L.kh, L.kw),
                                    dtype=L.dtype, stride=L.stride, pads=L.pads, dilation=L.dilation,
                                    out_pad=L.out_pad, groups=L.groups, act=L.act, has_bias=L.bias)
    ho, wo = conv.conv_transpose_output_shape(p)
    need = conv.conv_transpose_scratch_bytes(p)
    es = 4 if L.dtype == "f32" else 2
    set_bytes = es * (L.n * L.c_in * L.h * L.w + L.c_in * (L.c_out // L.groups) * L.kh * L.kw + L.n * L.c_out * ho * wo)
    nsets = max(1, min(64, math.ceil(2 * L2_BYTES / set_bytes)))
    sets = []
    for i in range(nsets):
        t = {k: (v.to(dev) if v is not None else None) for k, v in make_transpose_inputs(L, seed_offset=i + 1).items()}
        t["y"] = torch.empty((L.n, L.c_out, ho, wo), dtype=t["x"].dtype, device=dev)
        sets.append(t)
    scratch = torch.empty(need, dtype=torch.uint8, device=dev)

    def step(i):
        t = sets[i % nsets]
        conv.conv_transpose_forward(p, t["x"], t["w"], t["bias"], None, t["y"], scratch, need)

    for i in range(max(warmup, nsets)):
        step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for i in range(steps):
            step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank).start()
    t_end = time.time() + 0.5
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    us = secs * 1e6 / steps
    fl = transpose_flops(L)
    rate = fl / (us / 1e6) / 1e12
    # 16-bit layers with one group run their Gemm on the tensor cores (mma.sync,
    # weight transpose + Gemm + col2im); the others on the CUDA cores in float32
    # (plus the widening of a 16-bit x)
    tc = L.dtype != "f32" and L.groups == 1
    peak = MMA_SYNC_PEAK_TFLOPS if tc else FFMA_PEAK_TFLOPS
    launches = 3 if (tc or L.dtype == "f32") else 4
    return {"value": aggregate(fl * steps, world, secs) / 1e12, "us": us, "clocks": clocks,
            "launches": launches * steps, "tensor_gemm": tc,
            "roofline": {"bound": "tensor" if tc else "alu", "achieved": round(rate, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(rate / peak, 4),
                         "traffic": profiled_traffic(L.name, "", "conv_pointwise.cu" if tc else "conv_ffma.cu"),
                         "tensor_or_alu_frac": round(rate / peak, 4)}}


def nested_layers(headline: str, args, world: int, rank: int, local_rank: int) -> list:
    """Every other workload layer, timed like the headline (graphs of
    back-to-back calls, inputs rotated past L2, events on the launching
    stream) with --layer-steps steps: one compact record each."""
    from workloads import LAYERS
    out = []
    for name in sorted(LAYERS):
        if name == headline:
            continue
        L = LAYERS[name]
        r = run_ours(L, args.layer_steps, args.warmup, world, rank, local_rank,
                     with_cpu_baseline=False, with_e2e=False)
        roof = r["roofline"]
        rec = {"layer": name, "workload": describe(L), "dtype": L.dtype, "variant": r["variant"],
               "steps": args.layer_steps, "us_per_call": roof["launch_us"],
               "tflops": round(r["value"], 3),
               "gbs": round(aggregate(layer_bytes(L) * args.layer_steps, world, r["secs"]) / 1e9, 1),
               "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic",
                                                 "tensor_or_alu_frac")},
               "gpu_launches": r["launches"], "sm_mhz": r["clocks"].get("sm_mhz"),
               "clock_reasons": r["clocks"].get("reasons")}
        out.append(rec)
    from workloads import INT_LAYERS, TRANSPOSE_LAYERS
    for name in sorted(INT_LAYERS) + sorted(TRANSPOSE_LAYERS):
        out.append(other_op_record(name, args, world, local_rank))
    return out


def other_op_record(name: str, args, world: int, local_rank: int) -> dict:
    """The record of one ConvInteger or ConvTranspose workload layer."""
    from workloads import INT_LAYERS, TRANSPOSE_LAYERS
    if name in INT_LAYERS:
        L = INT_LAYERS[name]
        r = run_integer(L, args.layer_steps, args.warmup, world, local_rank)
        return {"layer": name, "workload": L.description, "dtype": f"{L.x_type}x{L.w_type}->i32",
                "variant": "conv_integer dp4a (unfold + weights + product)", "steps": args.layer_steps,
                "us_per_call": round(r["us"], 3), "tops": round(r["value"], 3), "roofline": r["roofline"],
                "gpu_launches": r["launches"], "sm_mhz": r["clocks"].get("sm_mhz"),
                "clock_reasons": r["clocks"].get("reasons")}
    L = TRANSPOSE_LAYERS[name]
    r = run_transpose(L, args.layer_steps, args.warmup, world, local_rank)
    return {"layer": name, "workload": L.description, "dtype": L.dtype,
            "variant": ("conv_transpose (weight transpose + tensor-core Gemm (mma.sync) + gathering col2im)"
                        if r["tensor_gemm"] else
                        "conv_transpose (weight transpose + float32 CUDA-core Gemm + gathering col2im)"),
            "steps": args.layer_steps, "us_per_call": round(r["us"], 3), "tflops": round(r["value"], 3),
            "roofline": r["roofline"], "gpu_launches": r["launches"], "sm_mhz": r["clocks"].get("sm_mhz"),
            "clock_reasons": r["clocks"].get("reasons")}


# ---- main ----------------------------------------------------------------
def describe(L) -> str:
    return L.description or L.name


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--layer-steps", type=int, default=300,
                    help="steps per nested layer of the default run")
    ap.add_argument("--no-layers", action="store_true",
                    help="the headline layer only (no nested per-layer rates)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layer", default=HEADLINE)
    ap.add_argument("--layers", default=None, help="'all': one line per workload layer")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="eager launches only, no e2e / CPU baseline (for profiler captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from workloads import INT_LAYERS, LAYERS, TRANSPOSE_LAYERS
    rank, world, local_rank = dist_env()
    names = sorted(LAYERS) if args.layers == "all" else [args.layer]
    other_op = args.layer in INT_LAYERS or args.layer in TRANSPOSE_LAYERS
    if other_op and args.impl != "ours":
        ap.error("--impl reference times the Conv layers only")

    if args.impl == "reference":
        if rank != 0:
            return 0
        for name in names:
            L = LAYERS[name]
            r = run_reference(L, args.steps, args.warmup)
            line = {"metric": METRIC, "value": r["value"], "unit": "TFLOP/s", "n_gpus": args.gpus,
                    "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": r["secs"] * 1e3 / args.steps, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
                    "data": "synthetic (seeded)",
                    "config": {"workload": describe(L), "layer": L.name,
                               "sample_outputs_per_step": r["per_step"],
                               "outputs_per_batch": r["total"]},
                    "cpu_baseline": {"value": r["value"], "unit": "TFLOP/s", "cores": r["cores"],
                                     "kind": "oracle",
                                     "sample": f"{r['per_step']} random outputs of one batch per step"},
                    "e2e": {"value": r["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if other_op:
        # one ConvInteger / ConvTranspose layer on its own (for profiler captures): its record only
        rec = other_op_record(args.layer, args, world, local_rank)
        if rank == 0:
            print(json.dumps(rec), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return 0
    nested = args.layers != "all" and not args.quick and not args.no_layers
    for name in names:
        L = LAYERS[name]
        r = run_ours(L, args.steps, args.warmup, world, rank, local_rank,
                     with_cpu_baseline=(rank == 0 and world == 1 and not args.no_cpu_baseline
                                        and not args.quick),
                     with_e2e=not args.quick, quick=args.quick)
        if rank != 0:
            continue
        line = {"metric": METRIC, "value": round(r["value"], 4), "unit": "TFLOP/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": r["secs"] * 1e3 / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": L.dtype,
                "data": "synthetic (seeded; the layer's shapes and value distributions; random weights)",
                "config": {"workload": describe(L), "layer": L.name, "global_batch": L.n * world,
                           "accumulate": "f32", "variant": r["variant"],
                           "l2": (f"inputs larger than L2: {r['nsets']} rotating sets of "
                                  f"{r['set_bytes'] / 1e6:.2f} MB"
                                  if r["nsets"] * r["set_bytes"] > L2_BYTES else
                                  f"L2-resident: {r['nsets']} rotating sets of "
                                  f"{r['set_bytes'] / 1e6:.3f} MB total below L2"),
                           "timing": ("eager launches" if args.quick else
                                      f"CUDA graphs of {r['chunk']} back-to-back steps"),
                           "parallelism": f"replicas x{world}"},
                "roofline": r["roofline"], "gpu_launches": r["launches"], "clocks": r["clocks"],
                "e2e": r.get("e2e")}
        if "cpu_baseline" in r:
            line["cpu_baseline"] = r["cpu_baseline"]
        if nested:
            line["layers"] = nested_layers(name, args, world, rank, local_rank)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
