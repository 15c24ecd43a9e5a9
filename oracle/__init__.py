"""CPU oracle for the INT8 NCxHWx<32> Conv2d forward pass -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline and
reference legs of ``bench.py`` may import this package.  The product library never calls it and
shares no code with it: the convolution, the epilogue and the layout
transforms here are written from their definitions, independently of the
CUDA kernels they check.

* ``conv_oracle.c`` -- direct convolution on NCHW/KCRS int8 with int64
  accumulation and the fp32 clamp epilogue (see its header for the passages
  it follows).  Compiled with gcc on first use (or by ``build()``).
* the layout helpers below -- NCHW <-> NCxHWx<32> and KCRS <-> CxRSKx<32>
  written as reshapes/transposes of the layouts' definitions (page 1's
  CUTLASS configuration names the layouts; the interleaved formula is the
  plain reading of their names: 32 consecutive channels per pixel).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}

INTERLEAVE = 32


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("N", "C", "H", "W", "K", "R", "S", "pad_h", "pad_w",
                 "stride_h", "stride_w", "dil_h", "dil_w")]


def lib_path(mutation: int = 0) -> str:
    name = "liboracle.so" if mutation == 0 else f"liboracle_mut{mutation}.so"
    return os.path.join(_BUILD, name)


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile the oracle (or one planted-mistake variant) with gcc."""
    out = lib_path(mutation)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", f"-DORACLE_MUTATION={mutation}",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutation: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutation not in _libs:
            lib = ctypes.CDLL(build(mutation))
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_out_extent.restype = i64
            lib.oracle_out_extent.argtypes = [i64] * 5
            lib.oracle_conv2d_acc.restype = ctypes.c_int
            lib.oracle_conv2d_acc.argtypes = [p, p, p, ctypes.POINTER(_Shape), ctypes.c_int]
            lib.oracle_conv2d_acc_points.restype = ctypes.c_int
            lib.oracle_conv2d_acc_points.argtypes = [p, p, ctypes.POINTER(_Shape), p, i64, p]
            lib.oracle_requantize.restype = ctypes.c_int
            lib.oracle_requantize.argtypes = [p, i64, ctypes.c_float, p]
            lib.oracle_requantize_channels.restype = ctypes.c_int
            lib.oracle_requantize_channels.argtypes = [p, i64, i64, i64, ctypes.c_float, p, p, ctypes.c_int, p]
            lib.oracle_conv2d_f64.restype = ctypes.c_int
            lib.oracle_conv2d_f64.argtypes = [p, p, p, p, p, ctypes.POINTER(_Shape), ctypes.c_int]
            lib.oracle_conv2d_f64_points.restype = ctypes.c_int
            lib.oracle_conv2d_f64_points.argtypes = [p, p, p, ctypes.POINTER(_Shape), p, i64, p, p]
            lib.oracle_mutation_id.restype = ctypes.c_int
            _libs[mutation] = lib
        return _libs[mutation]


class Oracle:
    """Handle on one compiled oracle variant (0 = the real oracle)."""

    def __init__(self, mutation: int = 0):
        self.mutation = mutation
        self.lib = _lib(mutation)

    # -- output size (page 4, first analysis paragraph) -------------------
    def out_extent(self, size, pad, dil, k, stride) -> int:
        return int(self.lib.oracle_out_extent(size, pad, dil, k, stride))

    def out_size(self, shape) -> tuple[int, int]:
        N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
        return self.out_extent(H, ph, dh, R, sh), self.out_extent(W, pw, dw, S, sw)

    # -- direct convolution ------------------------------------------------
    @staticmethod
    def _shape(shape) -> _Shape:
        return _Shape(*[int(v) for v in shape])

    def conv_acc(self, x_nchw: np.ndarray, f_kcrs: np.ndarray, shape, threads: int | None = None) -> np.ndarray:
        """int64 accumulators, NKPQ, of the direct convolution."""
        N, C, H, W, K, R, S = shape[:7]
        x = np.ascontiguousarray(x_nchw, dtype=np.int8)
        f = np.ascontiguousarray(f_kcrs, dtype=np.int8)
        assert x.shape == (N, C, H, W) and f.shape == (K, C, R, S)
        P, Q = self.out_size(shape)
        acc = np.zeros((N, K, max(P, 0), max(Q, 0)), dtype=np.int64)
        if threads is None:
            threads = os.cpu_count() or 1
        sh = self._shape(shape)
        rc = self.lib.oracle_conv2d_acc(x.ctypes.data, f.ctypes.data, acc.ctypes.data, ctypes.byref(sh), threads)
        if rc != 0:
            raise ValueError(f"oracle_conv2d_acc failed ({rc})")
        return acc

    def conv_acc_points(self, x_nchw, f_kcrs, shape, pts: np.ndarray) -> np.ndarray:
        """int64 accumulators at rows (n, k, p, q) of ``pts``."""
        x = np.ascontiguousarray(x_nchw, dtype=np.int8)
        f = np.ascontiguousarray(f_kcrs, dtype=np.int8)
        pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
        out = np.zeros(pts.shape[0], dtype=np.int64)
        sh = self._shape(shape)
        rc = self.lib.oracle_conv2d_acc_points(x.ctypes.data, f.ctypes.data, ctypes.byref(sh),
                                               pts.ctypes.data, pts.shape[0], out.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle_conv2d_acc_points failed ({rc})")
        return out

    # -- fp32 direct convolution (page 4), evaluated in double -------------
    def conv_f64(self, x_nchw, w_kcrs, shape, bias=None, threads: int | None = None):
        """(y, mag): NKPQ float64 outputs bias[k] + sum x*w of fp32 inputs, and
        the magnitude sums |bias[k]| + sum |x*w| that bound fp32 rounding."""
        N, C, H, W, K, R, S = shape[:7]
        x = np.ascontiguousarray(x_nchw, dtype=np.float32)
        w = np.ascontiguousarray(w_kcrs, dtype=np.float32)
        assert x.shape == (N, C, H, W) and w.shape == (K, C, R, S)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32).reshape(K)
        P, Q = self.out_size(shape)
        y = np.zeros((N, K, max(P, 0), max(Q, 0)), dtype=np.float64)
        mag = np.zeros_like(y)
        sh = self._shape(shape)
        rc = self.lib.oracle_conv2d_f64(x.ctypes.data, w.ctypes.data, None if b is None else b.ctypes.data,
                                        y.ctypes.data, mag.ctypes.data, ctypes.byref(sh),
                                        threads or (os.cpu_count() or 1))
        if rc != 0:
            raise ValueError(f"oracle_conv2d_f64 failed ({rc})")
        return y, mag

    def conv_f64_points(self, x_nchw, w_kcrs, shape, pts, bias=None):
        """(y, mag) at rows (n, k, p, q) of ``pts``."""
        K = shape[4]
        x = np.ascontiguousarray(x_nchw, dtype=np.float32)
        w = np.ascontiguousarray(w_kcrs, dtype=np.float32)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32).reshape(K)
        pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
        y = np.zeros(pts.shape[0], dtype=np.float64)
        mag = np.zeros_like(y)
        sh = self._shape(shape)
        rc = self.lib.oracle_conv2d_f64_points(x.ctypes.data, w.ctypes.data, None if b is None else b.ctypes.data,
                                               ctypes.byref(sh), pts.ctypes.data, pts.shape[0], y.ctypes.data,
                                               mag.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle_conv2d_f64_points failed ({rc})")
        return y, mag

    def f32_error_bound(self, mag, terms: int):
        """Largest difference between the exact sum and any fp32 evaluation of
        a dot product of ``terms`` products plus the bias, in any order, whose
        magnitude sum is ``mag``: gamma_{terms+1} * mag, gamma_n = n*u/(1-n*u)
        with the single-precision unit roundoff u = 2^-24 (the standard bound
        for a dot product whose products and sums are each rounded once; a
        fused multiply-add only rounds less).  Mutations 17 and 18 (planted
        mistakes for the pin test) use u = 2^-23 and gamma_terms."""
        u = 2.0 ** -23 if self.mutation == 17 else 2.0 ** -24
        n = terms if self.mutation == 18 else terms + 1
        return (n * u / (1.0 - n * u)) * np.asarray(mag, dtype=np.float64)

    # -- epilogue (page 1: LinearCombinationClamp, alpha only) -------------
    def requantize(self, acc: np.ndarray, alpha: float) -> np.ndarray:
        a = np.ascontiguousarray(acc, dtype=np.int64)
        y = np.zeros(a.shape, dtype=np.int8)
        rc = self.lib.oracle_requantize(a.ctypes.data, a.size, ctypes.c_float(alpha), y.ctypes.data)
        if rc == 2:
            raise OverflowError("accumulator outside int32")
        if rc != 0:
            raise ValueError(f"oracle_requantize failed ({rc})")
        return y

    def conv2d_fprop(self, x_nchw, f_kcrs, shape, alpha: float, threads: int | None = None):
        """(int8 NKPQ output, int64 NKPQ accumulators)."""
        acc = self.conv_acc(x_nchw, f_kcrs, shape, threads)
        return self.requantize(acc, alpha), acc

    # -- per-output-channel epilogue: scale, bias, ReLU, clamp -------------
    def requantize_channels(self, acc_nkpq: np.ndarray, alpha: float, alpha_k=None, bias_k=None,
                            relu: bool = False) -> np.ndarray:
        """int8 NKPQ output of clamp(rint(relu(alpha_k*float(acc) + bias_k)))."""
        a = np.ascontiguousarray(acc_nkpq, dtype=np.int64)
        N, K = a.shape[0], a.shape[1]
        PQ = int(np.prod(a.shape[2:])) if a.ndim > 2 else 1
        ak = None if alpha_k is None else np.ascontiguousarray(alpha_k, dtype=np.float32).reshape(K)
        bk = None if bias_k is None else np.ascontiguousarray(bias_k, dtype=np.float32).reshape(K)
        y = np.zeros(a.shape, dtype=np.int8)
        rc = self.lib.oracle_requantize_channels(a.ctypes.data, N, K, PQ, ctypes.c_float(alpha),
                                                 None if ak is None else ak.ctypes.data,
                                                 None if bk is None else bk.ctypes.data, int(bool(relu)),
                                                 y.ctypes.data)
        if rc == 2:
            raise OverflowError("accumulator outside int32")
        if rc != 0:
            raise ValueError(f"oracle_requantize_channels failed ({rc})")
        return y


# -- layouts ---------------------------------------------------------------
# NCxHWx<32>: element (n, c, h, w) at (((n*C/32 + c/32)*H + h)*W + w)*32 + c%32.
# CxRSKx<32>: element (k, c, r, s) at ((((c/32)*R + r)*S + s)*K + k)*32 + c%32.

def nchw_to_ncxhwx32(a: np.ndarray) -> np.ndarray:
    N, C, H, W = a.shape
    assert C % INTERLEAVE == 0
    return np.ascontiguousarray(a.reshape(N, C // 32, 32, H, W).transpose(0, 1, 3, 4, 2))


def ncxhwx32_to_nchw(a: np.ndarray, N: int, C: int, H: int, W: int) -> np.ndarray:
    v = a.reshape(N, C // 32, H, W, 32)
    return np.ascontiguousarray(v.transpose(0, 1, 4, 2, 3).reshape(N, C, H, W))


def kcrs_to_cxrskx32(f: np.ndarray) -> np.ndarray:
    K, C, R, S = f.shape
    assert C % INTERLEAVE == 0
    return np.ascontiguousarray(f.reshape(K, C // 32, 32, R, S).transpose(1, 3, 4, 0, 2))


def cxrskx32_to_kcrs(a: np.ndarray, K: int, C: int, R: int, S: int) -> np.ndarray:
    v = a.reshape(C // 32, R, S, K, 32)
    return np.ascontiguousarray(v.transpose(3, 0, 4, 1, 2).reshape(K, C, R, S))
