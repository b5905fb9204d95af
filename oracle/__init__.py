"""The CPU oracle for the forward 2-D convolution -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package never imports the library: the two share no code.

Contents
  * ``conv2d`` / ``conv2d_at``: the plain nested-loop definition (C, built with
    gcc into ``oracle/_build``), double accumulation, float32 epilogue.  See the
    header of ``conv_oracle.c`` for the passages it follows.
  * ``im2col.py``: a second, independent brute force (unfold, then one matrix
    product per group), written in numpy ("Convolutions", sections 2.4 and 3).
  * ``arith.py``: output size, MAC and parameter counts as closed forms
    ("Convolutions", sections 2.1 and 2.3).
  * number-format helpers: exact half / bfloat16 decoding and round-to-even
    encoding, used by the parity checks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_SRC_INT = os.path.join(_HERE, "conv_integer_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}

ACTIVATIONS = ("identity", "relu", "silu", "sigmoid", "tanh", "hard_swish",
               "hard_sigmoid", "clip", "leaky_relu")
_ACT_CODE = {name: i for i, name in enumerate(ACTIVATIONS)}
DTYPES = ("f32", "f16", "bf16")
_DT_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def library_path(mutant: int = 0) -> str:
    name = "libconv_oracle.so" if mutant == 0 else f"libconv_oracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the C oracle with gcc (no fused multiply-add, so the float32
    epilogue rounds each step on every host).  ``mutant`` > 0 plants one
    deliberate mistake; the pin tests use those builds to show they catch it."""
    out = library_path(mutant)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_INT))
    if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", f"-DORACLE_MUTANT={mutant}", _SRC, _SRC_INT, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutant in _libs:
            return _libs[mutant]
        lib = ctypes.CDLL(build(mutant))
        i64p = ctypes.POINTER(ctypes.c_int64)
        vp = ctypes.c_void_p
        lib.oracle_conv2d.argtypes = [i64p, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
        lib.oracle_conv2d.restype = ctypes.c_int
        lib.oracle_conv2d_at.argtypes = [i64p, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                         ctypes.c_int, vp, vp, vp, vp, i64p, ctypes.c_int64,
                                         vp, vp, vp, vp, ctypes.c_int]
        lib.oracle_conv2d_at.restype = ctypes.c_int
        lib.oracle_output_extent.argtypes = [ctypes.c_int64] * 6
        lib.oracle_output_extent.restype = ctypes.c_int64
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_float_to_half.argtypes = [ctypes.c_float]
        lib.oracle_float_to_half.restype = ctypes.c_uint16
        lib.oracle_float_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_float_to_bf16.restype = ctypes.c_uint16
        lib.oracle_activation.argtypes = [ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                          ctypes.c_float]
        lib.oracle_activation.restype = ctypes.c_float
        lib.oracle_mutant.restype = ctypes.c_int
        lib.oracle_conv_integer.argtypes = [i64p, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_int32,
                                            ctypes.POINTER(ctypes.c_int32), ctypes.c_int, i64p,
                                            ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
        lib.oracle_conv_integer.restype = ctypes.c_int
        lib.oracle_transpose_extent.argtypes = [ctypes.c_int64] * 7
        lib.oracle_transpose_extent.restype = ctypes.c_int64
        lib.oracle_conv_transpose2d.argtypes = [i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                                ctypes.c_float, ctypes.c_float, ctypes.c_int, vp, vp, vp, vp,
                                                i64p, ctypes.c_int64, vp, vp, vp, vp, ctypes.c_int]
        lib.oracle_conv_transpose2d.restype = ctypes.c_int
        _libs[mutant] = lib
        return lib


class Oracle:
    """Handle on one build of the C oracle (the real one, or a planted mutant)."""

    def __init__(self, mutant: int = 0):
        self.lib = _load(mutant)
        self.mutant = mutant

    # --- closed forms -------------------------------------------------------
    def output_extent(self, size, k, pad_begin, pad_end, stride=1, dilation=1) -> int:
        return int(self.lib.oracle_output_extent(size, k, pad_begin, pad_end, stride, dilation))

    def activation(self, act: str, t: float, alpha: float = 0.0, beta: float = 0.0) -> float:
        return float(self.lib.oracle_activation(_ACT_CODE[act], t, alpha, beta))

    def half_to_double(self, bits: int) -> float:
        return float(self.lib.oracle_half_to_double(bits))

    def bf16_to_double(self, bits: int) -> float:
        return float(self.lib.oracle_bf16_to_double(bits))

    def float_to_half(self, f: float) -> int:
        return int(self.lib.oracle_float_to_half(f))

    def float_to_bf16(self, f: float) -> int:
        return int(self.lib.oracle_float_to_bf16(f))

    # --- the convolution ----------------------------------------------------
    def conv2d(self, x, w, bias=None, residual=None, *, dtype="f32", stride=(1, 1),
               pads=(0, 0, 0, 0), dilation=(1, 1), groups=1, act="identity",
               alpha=0.0, beta=0.0, nthreads=None, index=None):
        """Evaluate the definition.

        x: (N, Cin, H, W) and w: (Cout, Cin/groups, kh, kw) numpy arrays --
        float32 for dtype "f32", uint16 bit patterns for "f16" / "bf16".
        bias: (Cout,), residual: (N, Cout, Ho, Wo), same element type.
        pads are ONNX order (top, left, bottom, right).
        index: optional 1-D int64 array of NCHW linear output indices; then
        only those outputs are computed (flat arrays of len(index) returned).

        Returns dict(y=..., t=float32 epilogue result, acc=double sum,
        scale=double sum of |w x|) with shape (N, Cout, Ho, Wo) or (len(index),).
        """
        geom, ho, wo = self.geometry(x.shape, w.shape, stride, pads, dilation, groups)
        want = np.float32 if dtype == "f32" else np.uint16
        arrs = [np.ascontiguousarray(a) if a is not None else None
                for a in (x, w, bias, residual)]
        for a in arrs:
            if a is not None and a.dtype != want:
                raise TypeError(f"oracle operand dtype {a.dtype}, expected {want} for {dtype}")
        n, cout = x.shape[0], w.shape[0]
        if arrs[2] is not None and arrs[2].shape != (cout,):
            raise ValueError("bias shape")
        if arrs[3] is not None and arrs[3].shape != (n, cout, ho, wo):
            raise ValueError("residual shape")
        shape = (n, cout, ho, wo) if index is None else (len(index),)
        y = np.empty(shape, dtype=want)
        t = np.empty(shape, dtype=np.float32)
        acc = np.empty(shape, dtype=np.float64)
        scale = np.empty(shape, dtype=np.float64)
        nthreads = nthreads or os.cpu_count() or 1
        g = (ctypes.c_int64 * 16)(*geom)
        ptr = lambda a: a.ctypes.data if a is not None else None
        common = (g, _ACT_CODE[act], alpha, beta, _DT_CODE[dtype],
                  ptr(arrs[0]), ptr(arrs[1]), ptr(arrs[2]), ptr(arrs[3]))
        if index is None:
            rc = self.lib.oracle_conv2d(*common, ptr(y), ptr(t), ptr(acc), ptr(scale), nthreads)
        else:
            idx = np.ascontiguousarray(index, dtype=np.int64)
            rc = self.lib.oracle_conv2d_at(
                *common, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(idx),
                ptr(y), ptr(t), ptr(acc), ptr(scale), nthreads)
        if rc != 0:
            raise ValueError("geometry outside the definition")
        return {"y": y, "t": t, "acc": acc, "scale": scale}

    def transpose_extent(self, size, k, pad_begin, pad_end, stride=1, dilation=1, out_pad=0) -> int:
        return int(self.lib.oracle_transpose_extent(size, k, pad_begin, pad_end, stride, dilation, out_pad))

    def conv_transpose2d(self, x, w, bias=None, residual=None, *, dtype="f32", stride=(1, 1),
                         pads=(0, 0, 0, 0), dilation=(1, 1), out_pad=(0, 0), groups=1, act="identity",
                         alpha=0.0, beta=0.0, nthreads=None, index=None):
        """The transposed convolution (ONNX ConvTranspose) by its gathering
        definition (see conv_oracle.c).  x: (N, Cin, H, W); w: (Cin, Cout/groups,
        kh, kw); element types and the returned dict as for conv2d."""
        n, cin, h, wd = x.shape
        cin_w, mg, kh, kw = w.shape
        if cin_w != cin or cin % groups:
            raise ValueError("weights [Cin][Cout/groups][kh][kw]")
        cout = mg * groups
        pt, pl, pb, pr = pads
        ho = self.transpose_extent(h, kh, pt, pb, stride[0], dilation[0], out_pad[0])
        wo = self.transpose_extent(wd, kw, pl, pr, stride[1], dilation[1], out_pad[1])
        if ho < 1 or wo < 1:
            raise ValueError("no output position")
        geom = [n, cin, h, wd, cout, kh, kw, pt, pl, pb, pr, stride[0], stride[1], dilation[0], dilation[1],
                groups]
        want = np.float32 if dtype == "f32" else np.uint16
        arrs = [np.ascontiguousarray(a) if a is not None else None for a in (x, w, bias, residual)]
        for a in arrs:
            if a is not None and a.dtype != want:
                raise TypeError(f"oracle operand dtype {a.dtype}, expected {want} for {dtype}")
        if arrs[3] is not None and arrs[3].shape != (n, cout, ho, wo):
            raise ValueError("residual shape")
        shape = (n, cout, ho, wo) if index is None else (len(index),)
        y = np.empty(shape, dtype=want)
        t = np.empty(shape, dtype=np.float32)
        acc = np.empty(shape, dtype=np.float64)
        scale = np.empty(shape, dtype=np.float64)
        g = (ctypes.c_int64 * 16)(*geom)
        ptr = lambda a: a.ctypes.data if a is not None else None
        idx = np.ascontiguousarray(index, dtype=np.int64) if index is not None else None
        rc = self.lib.oracle_conv_transpose2d(
            g, out_pad[0], out_pad[1], _ACT_CODE[act], alpha, beta, _DT_CODE[dtype], ptr(arrs[0]), ptr(arrs[1]),
            ptr(arrs[2]), ptr(arrs[3]),
            idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if idx is not None else None,
            len(idx) if idx is not None else 0, ptr(y), ptr(t), ptr(acc), ptr(scale),
            nthreads or os.cpu_count() or 1)
        if rc != 0:
            raise ValueError("geometry outside the definition")
        return {"y": y, "t": t, "acc": acc, "scale": scale}

    def conv_integer(self, x, w, x_zero=0, w_zero=0, *, stride=(1, 1), pads=(0, 0, 0, 0),
                     dilation=(1, 1), groups=1, nthreads=None, index=None):
        """ONNX ConvInteger by its definition ("Convolution, pooling and resize",
        ConvInteger): sum over the window of (x - x_zero) * (w - w_zero[co])
        in int32 with wrap-around, a padded tap being x_zero (adding nothing).

        x: (N, Cin, H, W) and w: (Cout, Cin/groups, kh, kw) numpy arrays of
        uint8 or int8 (any mix); x_zero: one value of x's type; w_zero: one
        value or Cout values of w's type.  Returns int32 (N, Cout, Ho, Wo),
        or the listed NCHW outputs (index) as a flat array."""
        for a in (x, w):
            if a.dtype not in (np.uint8, np.int8):
                raise TypeError(f"ConvInteger operands are uint8 or int8, not {a.dtype}")
        geom, ho, wo = self.geometry(x.shape, w.shape, stride, pads, dilation, groups)
        xs, ws = int(x.dtype == np.int8), int(w.dtype == np.int8)
        wz = np.atleast_1d(np.asarray(w_zero)).astype(np.int64)
        per_channel = wz.size > 1
        if per_channel and wz.size != w.shape[0]:
            raise ValueError("w_zero: one value or one per output channel")
        lo, hi = (-128, 127) if xs else (0, 255)
        if not lo <= int(x_zero) <= hi:
            raise ValueError("x_zero outside x's type")
        lo, hi = (-128, 127) if ws else (0, 255)
        if wz.min() < lo or wz.max() > hi:
            raise ValueError("w_zero outside w's type")
        wz32 = np.ascontiguousarray(wz, dtype=np.int32)
        xa, wa = np.ascontiguousarray(x), np.ascontiguousarray(w)
        n, cout = x.shape[0], w.shape[0]
        shape = (n, cout, ho, wo) if index is None else (len(index),)
        y = np.empty(shape, dtype=np.int32)
        g = (ctypes.c_int64 * 16)(*geom)
        i32p = ctypes.POINTER(ctypes.c_int32)
        idx = None
        if index is not None:
            idx = np.ascontiguousarray(index, dtype=np.int64)
        rc = self.lib.oracle_conv_integer(
            g, xs, ws, xa.ctypes.data, wa.ctypes.data, int(x_zero), wz32.ctypes.data_as(i32p),
            int(per_channel), idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if idx is not None else None,
            len(idx) if idx is not None else 0, y.ctypes.data_as(i32p), nthreads or os.cpu_count() or 1)
        if rc != 0:
            raise ValueError("geometry outside the definition")
        return y

    def geometry(self, xshape, wshape, stride, pads, dilation, groups):
        n, cin, h, w_ = xshape
        cout, cin_g, kh, kw = wshape
        if cin_g * groups != cin:
            raise ValueError("weight channels x groups != input channels")
        pt, pl, pb, pr = pads
        ho = self.output_extent(h, kh, pt, pb, stride[0], dilation[0])
        wo = self.output_extent(w_, kw, pl, pr, stride[1], dilation[1])
        geom = [n, cin, h, w_, cout, kh, kw, pt, pl, pb, pr,
                stride[0], stride[1], dilation[0], dilation[1], groups]
        return geom, ho, wo


def to_float64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact decode of an operand array to float64 (half / bfloat16 bit
    patterns by their IEEE / bfloat16 definitions)."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    bits = a.astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def ulp(y: np.ndarray, dtype: str) -> np.ndarray:
    """One unit in the last place of the element type at |y| (the spacing of
    representable values there; the subnormal spacing below the normal range)."""
    mant_bits, min_exp = {"f32": (23, -126), "f16": (10, -14), "bf16": (7, -126)}[dtype]
    a = np.abs(np.asarray(y, dtype=np.float64))
    # zero and the subnormals share the spacing of the smallest normal binade
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 2.0 ** min_exp)))
    e = np.maximum(e, min_exp)
    return np.ldexp(1.0, (e - mant_bits).astype(np.int64))
