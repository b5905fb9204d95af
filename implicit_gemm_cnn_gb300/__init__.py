"""implicit_gemm_cnn_gb300 -- forward 2-D convolution (ONNX Conv semantics) on
NVIDIA GB300 (sm_103a).

A thin ctypes binding of the C ABI in ``include/conv.h`` (libconv.so, built
in-tree by ``implicit_gemm_cnn_gb300.build``).  The functions keep the C names
and only marshal arguments; every step of the computation runs in the
library's CUDA kernels.  PyTorch is used for device memory and streams.

    import torch, implicit_gemm_cnn_gb300 as conv
    y = conv.conv2d(x, w, bias, stride=2, pads=3, act="relu")   # x, w on cuda

The library must be built (``python -m implicit_gemm_cnn_gb300.build``); a
missing or unloadable library raises ``ConvLibraryError`` -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "ConvError", "ConvLibraryError", "ConvProblem", "ConvPlanInfo", "ACTIVATIONS", "DTYPES",
    "FLAG_FORCE_FFMA", "FLAG_NO_SPLIT_K", "FLAG_NO_WINDOW", "FLAG_NO_UNFOLD", "FLAG_FORCE_UNFOLD", "FLAG_WINOGRAD",
    "FLAG_NO_WINOGRAD", "FLAG_NO_DW_MMA", "FLAG_NO_PW_MMA", "FLAG_NO_CLUSTER_K", "VARIANTS", "conv_abi_version", "conv_status_string",
    "conv_output_shape", "conv_plan", "conv_scratch_bytes", "conv_describe_variant", "conv_describe_plan",
    "conv_forward", "conv_device_error", "conv_selftest_bounded_wait", "conv_forward_fixed_scratch",
    "FIXED_SCRATCH_BYTES",
    "conv_apply_auto_pad", "AUTO_PAD", "conv_scratch_bytes_per_image",
    "conv_integer_scratch_bytes", "conv_integer_forward", "conv_integer2d", "INT_TYPES",
    "ConvTransposeProblem", "make_transpose_problem", "conv_transpose_output_shape",
    "conv_transpose_scratch_bytes", "conv_transpose_forward", "conv_transpose2d",
    "make_problem", "conv2d", "HostPipeline", "library_path", "load",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libconv.so")

ACTIVATIONS = {"identity": 0, "relu": 1, "silu": 2, "sigmoid": 3, "tanh": 4, "hard_swish": 5,
               "hard_sigmoid": 6, "clip": 7, "leaky_relu": 8}
DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
VARIANTS = {0: "igemm_ffma", 1: "igemm_ffma_split_k", 2: "depthwise_halo", 3: "igemm_tcgen05",
            4: "igemm_tcgen05_window", 5: "winograd_f2x2_3x3", 6: "pointwise_mma"}
FIXED_SCRATCH_BYTES = 8 << 20  # CONV_FIXED_SCRATCH_BYTES
FLAG_FORCE_FFMA = 0x1
FLAG_NO_SPLIT_K = 0x2
FLAG_NO_WINDOW = 0x4
FLAG_NO_UNFOLD = 0x8
FLAG_FORCE_UNFOLD = 0x10
FLAG_WINOGRAD = 0x20
FLAG_NO_WINOGRAD = 0x40
FLAG_NO_DW_MMA = 0x80
FLAG_NO_PW_MMA = 0x4000
FLAG_NO_CLUSTER_K = 0x8000
SPLIT_K_SHIFT = 8
STATUS = {0: "CONV_OK", 1: "CONV_ERR_SHAPE", 2: "CONV_ERR_OVERFLOW", 3: "CONV_ERR_DTYPE",
          4: "CONV_ERR_ACT", 5: "CONV_ERR_NULL", 6: "CONV_ERR_SCRATCH", 7: "CONV_ERR_ALIAS",
          8: "CONV_ERR_DEVICE", 9: "CONV_ERR_CUDA", 10: "CONV_ERR_ARG"}


class ConvLibraryError(RuntimeError):
    """libconv.so is missing or cannot be loaded."""


class ConvError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        msg = f"{where}: {self.name}" if where else self.name
        try:
            msg += f" ({conv_status_string(status)})"
        except ConvLibraryError:
            pass
        super().__init__(msg)


class ConvProblem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "n", "c_in", "h", "w", "c_out", "kh", "kw", "pad_top", "pad_left", "pad_bottom",
        "pad_right", "stride_h", "stride_w", "dil_h", "dil_w", "groups")] + [
        ("act", ctypes.c_int32), ("act_alpha", ctypes.c_float), ("act_beta", ctypes.c_float),
        ("dtype", ctypes.c_int32), ("has_bias", ctypes.c_int32), ("has_residual", ctypes.c_int32),
        ("flags", ctypes.c_uint32)]


class ConvTransposeProblem(ctypes.Structure):
    _fields_ = [("conv", ConvProblem), ("out_pad_h", ctypes.c_int64), ("out_pad_w", ctypes.c_int64)]


class ConvPlanInfo(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("ho", ctypes.c_int64), ("wo", ctypes.c_int64), ("gemm_m", ctypes.c_int64),
                ("gemm_n", ctypes.c_int64), ("gemm_k", ctypes.c_int64), ("ctas", ctypes.c_int64),
                ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("scratch_bytes", ctypes.c_uint64)]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["variant_name"] = VARIANTS.get(self.variant, "unknown")
        return d


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libconv.so (once).  Raises ConvLibraryError when it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ConvLibraryError(
                f"{_LIB_PATH} not found: build it with `python -m implicit_gemm_cnn_gb300.build`")
        try:
            lib = ctypes.CDLL(_LIB_PATH)
        except OSError as e:
            raise ConvLibraryError(f"cannot load {_LIB_PATH}: {e}") from e
        P = ctypes.POINTER
        vp = ctypes.c_void_p
        lib.conv_abi_version.restype = ctypes.c_int32
        lib.conv_status_string.argtypes = [ctypes.c_int]
        lib.conv_status_string.restype = ctypes.c_char_p
        lib.conv_output_shape.argtypes = [P(ConvProblem), P(ctypes.c_int64), P(ctypes.c_int64)]
        lib.conv_plan.argtypes = [P(ConvProblem), ctypes.c_int32, P(ConvPlanInfo)]
        lib.conv_scratch_bytes.argtypes = [P(ConvProblem), P(ctypes.c_size_t)]
        lib.conv_describe_variant.argtypes = [P(ConvProblem), ctypes.c_char_p, ctypes.c_size_t]
        lib.conv_describe_plan.argtypes = [P(ConvProblem), ctypes.c_int32, ctypes.c_char_p, ctypes.c_size_t]
        lib.conv_forward.argtypes = [P(ConvProblem), vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.conv_device_error.argtypes = [P(ctypes.c_uint32), ctypes.c_int32]
        lib.conv_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P(ctypes.c_uint32)]
        lib.conv_forward_fixed_scratch.argtypes = [P(ConvProblem), vp, vp, vp, vp, vp, vp]
        lib.conv_apply_auto_pad.argtypes = [P(ConvProblem), ctypes.c_int32]
        lib.conv_scratch_bytes_per_image.argtypes = [P(ConvProblem), P(ctypes.c_size_t)]
        lib.conv_transpose_output_shape.argtypes = [P(ConvTransposeProblem), P(ctypes.c_int64), P(ctypes.c_int64)]
        lib.conv_transpose_scratch_bytes.argtypes = [P(ConvTransposeProblem), P(ctypes.c_size_t)]
        lib.conv_transpose_forward.argtypes = [P(ConvTransposeProblem), vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.conv_integer_scratch_bytes.argtypes = [P(ConvProblem), ctypes.c_int32, ctypes.c_int32,
                                                   P(ctypes.c_size_t)]
        lib.conv_integer_forward.argtypes = [P(ConvProblem), ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp,
                                             ctypes.c_int32, vp, vp, ctypes.c_size_t, vp]
        for f in ("conv_output_shape", "conv_plan", "conv_scratch_bytes", "conv_describe_variant",
                  "conv_describe_plan", "conv_forward", "conv_device_error", "conv_selftest_bounded_wait",
                  "conv_forward_fixed_scratch", "conv_apply_auto_pad",
                  "conv_scratch_bytes_per_image", "conv_integer_scratch_bytes", "conv_integer_forward",
                  "conv_transpose_output_shape", "conv_transpose_scratch_bytes", "conv_transpose_forward"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise ConvError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


# ---- the C functions, same names --------------------------------------------
def conv_abi_version() -> int:
    return load().conv_abi_version()


def conv_status_string(status: int) -> str:
    return load().conv_status_string(status).decode()


def conv_output_shape(p: ConvProblem) -> tuple[int, int]:
    ho, wo = ctypes.c_int64(), ctypes.c_int64()
    _check(load().conv_output_shape(ctypes.byref(p), ctypes.byref(ho), ctypes.byref(wo)),
           "conv_output_shape")
    return ho.value, wo.value


AUTO_PAD = {"NOTSET": 0, "SAME_UPPER": 1, "SAME_LOWER": 2, "VALID": 3}


def conv_apply_auto_pad(p: ConvProblem, mode: str) -> ConvProblem:
    """Set p's pads from ONNX auto_pad `mode` (in place; p is returned)."""
    _check(load().conv_apply_auto_pad(ctypes.byref(p), AUTO_PAD[mode]), "conv_apply_auto_pad")
    return p


def conv_plan(p: ConvProblem, sm_count: int) -> dict:
    info = ConvPlanInfo()
    _check(load().conv_plan(ctypes.byref(p), sm_count, ctypes.byref(info)), "conv_plan")
    return info.as_dict()


def conv_scratch_bytes(p: ConvProblem) -> int:
    n = ctypes.c_size_t()
    _check(load().conv_scratch_bytes(ctypes.byref(p), ctypes.byref(n)), "conv_scratch_bytes")
    return n.value


def conv_scratch_bytes_per_image(p: ConvProblem) -> int:
    n = ctypes.c_size_t()
    _check(load().conv_scratch_bytes_per_image(ctypes.byref(p), ctypes.byref(n)), "conv_scratch_bytes_per_image")
    return n.value


def conv_describe_variant(p: ConvProblem) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(load().conv_describe_variant(ctypes.byref(p), buf, len(buf)), "conv_describe_variant")
    return buf.value.decode()


def conv_describe_plan(p: ConvProblem, sm_count: int) -> str:
    """conv_describe_variant's description for a device with ``sm_count`` SMs,
    computed on the host only."""
    buf = ctypes.create_string_buffer(512)
    _check(load().conv_describe_plan(ctypes.byref(p), int(sm_count), buf, len(buf)), "conv_describe_plan")
    return buf.value.decode()


def conv_forward(p: ConvProblem, x, w, bias, residual, y, scratch=None, scratch_bytes: int = 0,
                 stream=None) -> None:
    """Enqueue the convolution.  Tensors (anything with .data_ptr()) or raw
    device addresses; ``stream`` a torch.cuda.Stream, a raw cudaStream_t, or
    None for the current torch stream (the legacy default stream without torch)."""
    if stream is None:
        try:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        except Exception:  # noqa: BLE001 - no torch / no CUDA: the legacy default stream
            stream = 0
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    _check(load().conv_forward(ctypes.byref(p), _ptr(x), _ptr(w), _ptr(bias), _ptr(residual),
                               _ptr(y), _ptr(scratch), scratch_bytes, stream or None),
           "conv_forward")


def conv_forward_fixed_scratch(p: ConvProblem, x, w, bias, residual, y, stream=None) -> None:
    """conv_forward with the split-k scratch in the library's own fixed device
    array (FIXED_SCRATCH_BYTES) instead of caller memory: for callers that
    cannot allocate device memory.  The first call on a device sets the array
    up (before any stream capture); calls that overlap on the GPU race on it."""
    if stream is None:
        try:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        except Exception:  # noqa: BLE001 - no torch / no CUDA: the legacy default stream
            stream = 0
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    _check(load().conv_forward_fixed_scratch(ctypes.byref(p), _ptr(x), _ptr(w), _ptr(bias),
                                             _ptr(residual), _ptr(y), stream or None),
           "conv_forward_fixed_scratch")


def make_transpose_problem(x_shape, w_shape, *, dtype="f32", stride=1, pads=0, dilation=1, out_pad=0,
                           groups=1, act="identity", alpha=0.0, beta=0.0, has_bias=False,
                           has_residual=False, flags=0) -> ConvTransposeProblem:
    """x (N, Cin, H, W); w (Cin, Cout/groups, kh, kw).  ``flags``:
    FLAG_NO_PW_MMA keeps a 16-bit layer's Gemm on the CUDA cores."""
    n, c_in, h, w = (int(v) for v in x_shape)
    cin_w, mg, kh, kw = (int(v) for v in w_shape)
    if cin_w != c_in:
        raise ValueError("ConvTranspose weights are [Cin][Cout/groups][kh][kw]")
    q = make_problem((n, c_in, h, w), (mg * int(groups), c_in // int(groups), kh, kw), dtype=dtype,
                     stride=stride, pads=pads, dilation=dilation, groups=groups, act=act, alpha=alpha,
                     beta=beta, has_bias=has_bias, has_residual=has_residual, flags=flags)
    oph, opw = _pair(out_pad)
    return ConvTransposeProblem(q, oph, opw)


def conv_transpose_output_shape(p: ConvTransposeProblem) -> tuple[int, int]:
    ho, wo = ctypes.c_int64(), ctypes.c_int64()
    _check(load().conv_transpose_output_shape(ctypes.byref(p), ctypes.byref(ho), ctypes.byref(wo)),
           "conv_transpose_output_shape")
    return ho.value, wo.value


def conv_transpose_scratch_bytes(p: ConvTransposeProblem) -> int:
    n = ctypes.c_size_t()
    _check(load().conv_transpose_scratch_bytes(ctypes.byref(p), ctypes.byref(n)), "conv_transpose_scratch_bytes")
    return n.value


def conv_transpose_forward(p: ConvTransposeProblem, x, w, bias, residual, y, scratch, scratch_bytes: int,
                           stream=None) -> None:
    if stream is None:
        try:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        except Exception:  # noqa: BLE001 - no torch / no CUDA: the legacy default stream
            stream = 0
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    _check(load().conv_transpose_forward(ctypes.byref(p), _ptr(x), _ptr(w), _ptr(bias), _ptr(residual), _ptr(y),
                                         _ptr(scratch), scratch_bytes, stream or None), "conv_transpose_forward")


def conv_transpose2d(x, w, bias=None, residual=None, *, stride=1, pads=0, dilation=1, out_pad=0, groups=1,
                     act="identity", alpha=0.0, beta=0.0, out=None, scratch=None, stream=None, flags=0):
    """ConvTranspose on CUDA tensors (w [Cin][Cout/groups][kh][kw]); allocates
    y and scratch with torch unless given."""
    import torch
    dt = _dtype_name(x)
    p = make_transpose_problem(x.shape, w.shape, dtype=dt, stride=stride, pads=pads, dilation=dilation,
                               out_pad=out_pad, groups=groups, act=act, alpha=alpha, beta=beta,
                               has_bias=bias is not None, has_residual=residual is not None, flags=flags)
    ho, wo = conv_transpose_output_shape(p)
    if out is None:
        out = torch.empty((p.conv.n, p.conv.c_out, ho, wo), dtype=x.dtype, device=x.device)
    need = conv_transpose_scratch_bytes(p)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=x.device)
    conv_transpose_forward(p, x, w, bias, residual, out, scratch, scratch.numel() * scratch.element_size(), stream)
    return out


INT_TYPES = {"u8": 0, "i8": 1}


def conv_integer_scratch_bytes(p: ConvProblem, x_type: str, w_type: str) -> int:
    n = ctypes.c_size_t()
    _check(load().conv_integer_scratch_bytes(ctypes.byref(p), INT_TYPES[x_type], INT_TYPES[w_type],
                                             ctypes.byref(n)), "conv_integer_scratch_bytes")
    return n.value


def conv_integer_forward(p: ConvProblem, x_type: str, w_type: str, x, w, x_zero, w_zero, w_zero_count: int,
                         y, scratch, scratch_bytes: int, stream=None) -> None:
    """Enqueue ConvInteger (int32 output with wrap-around)."""
    if stream is None:
        try:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        except Exception:  # noqa: BLE001 - no torch / no CUDA: the legacy default stream
            stream = 0
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    _check(load().conv_integer_forward(ctypes.byref(p), INT_TYPES[x_type], INT_TYPES[w_type], _ptr(x), _ptr(w),
                                       _ptr(x_zero), _ptr(w_zero), int(w_zero_count), _ptr(y), _ptr(scratch),
                                       scratch_bytes, stream or None), "conv_integer_forward")


def conv_integer2d(x, w, x_zero, w_zero, *, stride=1, pads=0, dilation=1, groups=1, out=None, scratch=None,
                   stream=None, auto_pad="NOTSET"):
    """ConvInteger on CUDA tensors: x, w uint8 / int8 (NCHW / OIHW), x_zero a
    one-element tensor of x's type, w_zero one element or one per output
    channel of w's type.  Returns int32 y (allocated unless ``out``)."""
    import torch
    tn = {torch.uint8: "u8", torch.int8: "i8"}
    if x.dtype not in tn or w.dtype not in tn:
        raise TypeError("ConvInteger operands are uint8 or int8")
    if x_zero.dtype != x.dtype or w_zero.dtype != w.dtype or x_zero.numel() != 1:
        raise ValueError("zero points: one element of x's type; one or c_out elements of w's type")
    p = make_problem(x.shape, w.shape, stride=stride, pads=pads, dilation=dilation, groups=groups,
                     auto_pad=auto_pad)
    ho, wo = conv_output_shape(p)
    if out is None:
        out = torch.empty((p.n, p.c_out, ho, wo), dtype=torch.int32, device=x.device)
    need = conv_integer_scratch_bytes(p, tn[x.dtype], tn[w.dtype])
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=x.device)
    conv_integer_forward(p, tn[x.dtype], tn[w.dtype], x, w, x_zero, w_zero, w_zero.numel(), out, scratch,
                         scratch.numel() * scratch.element_size(), stream)
    return out


def conv_device_error(reset: bool = True) -> int:
    word = ctypes.c_uint32()
    _check(load().conv_device_error(ctypes.byref(word), 1 if reset else 0), "conv_device_error")
    return word.value


def conv_selftest_bounded_wait(limit_us: int = 1000) -> list[int]:
    """The five report words of the give-up-path self test (see include/conv.h)."""
    report = (ctypes.c_uint32 * 5)()
    _check(load().conv_selftest_bounded_wait(int(limit_us), report), "conv_selftest_bounded_wait")
    return list(report)



class HostPipeline:
    """conv2d over batches that live in (pinned) host memory, with the copies
    overlapped: the host->device copy of one batch, the convolution of the
    previous one and the device->host copy of the one before run at the same
    time on three CUDA streams, over two device buffers of x and of y used in
    turn.  Each batch's result is the one conv2d gives.  w, bias and residual
    are device tensors shared by every batch; the scratch is allocated once.

    ``run`` enqueues and returns; the caller's current stream waits for all of
    it, so a synchronize (or any later work on that stream) sees the results.
    """

    def __init__(self, x_shape, w, bias=None, residual=None, *, stride=1, pads=0, dilation=1, groups=1,
                 act="identity", alpha=0.0, beta=0.0, flags=0, auto_pad="NOTSET"):
        import torch
        self._torch = torch
        dt = _dtype_name(w)
        self.p = make_problem(tuple(x_shape), w.shape, dtype=dt, stride=stride, pads=pads, dilation=dilation,
                              groups=groups, act=act, alpha=alpha, beta=beta, has_bias=bias is not None,
                              has_residual=residual is not None, flags=flags, auto_pad=auto_pad)
        ho, wo = conv_output_shape(self.p)
        dev = w.device
        self.w, self.bias, self.residual = w, bias, residual
        self.x_dev = [torch.empty(tuple(x_shape), dtype=w.dtype, device=dev) for _ in range(2)]
        self.y_dev = [torch.empty((self.p.n, self.p.c_out, ho, wo), dtype=w.dtype, device=dev) for _ in range(2)]
        self.need = conv_scratch_bytes(self.p)
        self.scratch = torch.empty(self.need, dtype=torch.uint8, device=dev) if self.need else None
        self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_comp = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]
        self.turn = 0

    def run(self, x_hosts, y_hosts) -> None:
        torch = self._torch
        cur = torch.cuda.current_stream()
        for s in (self.s_in, self.s_comp, self.s_out):
            s.wait_stream(cur)
        for xh, yh in zip(x_hosts, y_hosts):
            b = self.turn
            self.turn ^= 1
            with torch.cuda.stream(self.s_in):
                if self.used[b]:
                    self.s_in.wait_event(self.ev_comp[b])  # the convolution that read x_dev[b] is done
                self.x_dev[b].copy_(xh, non_blocking=True)
                self.ev_in[b].record(self.s_in)
            self.s_comp.wait_event(self.ev_in[b])
            if self.used[b]:
                self.s_comp.wait_event(self.ev_out[b])  # y_dev[b] has been copied out
            conv_forward(self.p, self.x_dev[b], self.w, self.bias, self.residual, self.y_dev[b], self.scratch,
                         self.need, self.s_comp)
            self.ev_comp[b].record(self.s_comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(self.ev_comp[b])
                yh.copy_(self.y_dev[b], non_blocking=True)
                self.ev_out[b].record(self.s_out)
            self.used[b] = True
        for s in (self.s_in, self.s_comp, self.s_out):
            cur.wait_stream(s)


# ---- conveniences ---------------------------------------------------------
def _pair(v) -> tuple[int, int]:
    return (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))


def _pads(v) -> tuple[int, int, int, int]:
    if isinstance(v, int):
        return (v, v, v, v)
    v = tuple(int(t) for t in v)
    if len(v) == 2:
        return (v[0], v[1], v[0], v[1])
    return v  # ONNX order: top, left, bottom, right


def make_problem(x_shape, w_shape, *, dtype="f32", stride=1, pads=0, dilation=1, groups=1,
                 act="identity", alpha=0.0, beta=0.0, has_bias=False, has_residual=False,
                 flags=0, auto_pad="NOTSET") -> ConvProblem:
    n, c_in, h, w = (int(v) for v in x_shape)
    c_out, _, kh, kw = (int(v) for v in w_shape)
    sh, sw = _pair(stride)
    dh, dw = _pair(dilation)
    pt, pl, pb, pr = _pads(pads)
    p = ConvProblem(n, c_in, h, w, c_out, kh, kw, pt, pl, pb, pr, sh, sw, dh, dw, int(groups),
                    ACTIVATIONS[act], float(alpha), float(beta), DTYPES[dtype],
                    1 if has_bias else 0, 1 if has_residual else 0, int(flags))
    if auto_pad != "NOTSET":
        conv_apply_auto_pad(p, auto_pad)
    return p


_TORCH_DT = None


def _dtype_name(t) -> str:
    global _TORCH_DT
    import torch
    if _TORCH_DT is None:
        _TORCH_DT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
    if t.dtype not in _TORCH_DT:
        raise TypeError(f"unsupported element type {t.dtype}")
    return _TORCH_DT[t.dtype]


def conv2d(x, w, bias=None, residual=None, *, stride=1, pads=0, dilation=1, groups=1,
           act="identity", alpha=0.0, beta=0.0, out=None, scratch=None, flags=0, stream=None,
           auto_pad="NOTSET"):
    """y = act(conv(x, w) + bias + residual) on CUDA tensors (NCHW / OIHW,
    contiguous, one element type).  ``auto_pad`` (ONNX: SAME_UPPER, SAME_LOWER,
    VALID) replaces ``pads`` when set.  Allocates y (and the scratch the plan
    needs) with torch unless ``out`` / ``scratch`` are given."""
    import torch
    dt = _dtype_name(x)
    for t in (w, bias, residual, out):
        if t is not None and (t.dtype != x.dtype or not t.is_contiguous() or t.device != x.device):
            raise ValueError("operands must share x's element type and device and be contiguous")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous NCHW")
    p = make_problem(x.shape, w.shape, dtype=dt, stride=stride, pads=pads, dilation=dilation,
                     groups=groups, act=act, alpha=alpha, beta=beta, has_bias=bias is not None,
                     has_residual=residual is not None, flags=flags, auto_pad=auto_pad)
    ho, wo = conv_output_shape(p)
    if out is None:
        out = torch.empty((p.n, p.c_out, ho, wo), dtype=x.dtype, device=x.device)
    need = conv_scratch_bytes(p)
    if need and scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=x.device)
    conv_forward(p, x, w, bias, residual, out, scratch, scratch.numel() * scratch.element_size()
                 if scratch is not None else 0, stream)
    return out
