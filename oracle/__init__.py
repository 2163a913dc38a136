"""ctypes front end of the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference legs of ``bench.py`` import this package.  The CUDA
library and its Python binding never import it, and it imports nothing from
them: inputs arrive as numpy arrays of bf16 bit patterns (uint16), FP8
codes (uint8) and fp32.

The program is a list of op names, optionally with one numeric argument:
``alpha, bias, row_scale, residual, gelu_tanh, relu, silu, pair_swiglu[:g], pair_mul[:g],
gelu_tanh_grad, amax, store_bf16, store_e4m3, row_rms[:eps],
row_rms_unrounded[:eps], col_sum, dswiglu[:g], col_scale, row_dot``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from . import build as _build

_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("b_is_nk", ctypes.c_int),
        ("A", ctypes.c_void_p), ("lda", ctypes.c_int64),
        ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("B2", ctypes.c_void_p),
        ("alpha", ctypes.c_double),
        ("bias", ctypes.c_void_p), ("row_scale", ctypes.c_void_p),
        ("residual", ctypes.c_void_p), ("preact", ctypes.c_void_p),
        ("ld_aux", ctypes.c_int64),
        ("fp8_scale", ctypes.c_double),
        ("program", ctypes.c_char_p),
        ("a_type", ctypes.c_int), ("b_type", ctypes.c_int),
        ("a_scale_inv", ctypes.c_double), ("b_scale_inv", ctypes.c_double),
        ("col_scale", ctypes.c_void_p),
    ]


# Operand element types: bf16 bit patterns (uint16) or FP8 codes (uint8).
TYPES = {"bf16": 0, "e4m3": 1, "e5m2": 2}


def load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(_Problem)
        vp = ctypes.c_void_p
        lib.oracle_rows.argtypes = [P, vp, ctypes.c_int64, vp, vp, vp, vp, vp]
        lib.oracle_rows.restype = ctypes.c_int
        lib.oracle_cols.argtypes = [P, vp, ctypes.c_int64, vp, vp]
        lib.oracle_cols.restype = ctypes.c_int
        lib.oracle_out_cols.argtypes = [P]
        lib.oracle_out_cols.restype = ctypes.c_int
        for name in ("oracle_gelu_tanh", "oracle_gelu_tanh_grad", "oracle_silu", "oracle_silu_grad"):
            getattr(lib, name).argtypes = [ctypes.c_double]
            getattr(lib, name).restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_double_to_e4m3.argtypes = [ctypes.c_double]
        lib.oracle_double_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_rmsnorm_backward.argtypes = [ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_int64, vp,
                                                ctypes.c_int64, vp, vp, vp, vp, ctypes.c_int64, vp, vp]
        lib.oracle_rmsnorm_backward.restype = None
        lib.oracle_e5m2_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e5m2_to_double.restype = ctypes.c_double
        _lib = lib
    return _lib


def _u16(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as uint16 bit patterns")
    return a


def _operand(a, type_name):
    if a is None:
        return None
    if type_name == "bf16":
        return _u16(a)
    if type_name not in TYPES:
        raise ValueError("unknown operand type %r" % type_name)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("FP8 operands are passed as uint8 codes")
    return a


def _f32(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


@dataclass
class Problem:
    """One GEMM + epilogue problem in the oracle's terms.

    A: M x K bf16 bits (uint16) or FP8 codes (uint8, ``a_type`` "e4m3" or
    "e5m2"), row-major with row stride ``A.shape[1]``.
    B: K x N when ``b_is_nk`` is False, else N x K, of type ``b_type``.
    B2: optional second weight operand of B's shape; the accumulator then
    has 2 x B's columns, alternating between B and B2 in blocks of 128.
    a_scale_inv, b_scale_inv: per-tensor dequantisation factors; the
    accumulator is their product times A @ B.
    """
    A: np.ndarray
    B: np.ndarray
    program: Sequence[str]
    b_is_nk: bool = False
    alpha: float = 1.0
    bias: Optional[np.ndarray] = None
    row_scale: Optional[np.ndarray] = None
    residual: Optional[np.ndarray] = None
    preact: Optional[np.ndarray] = None
    fp8_scale: float = 1.0
    B2: Optional[np.ndarray] = None
    a_type: str = "bf16"
    b_type: str = "bf16"
    a_scale_inv: float = 1.0
    b_scale_inv: float = 1.0
    col_scale: Optional[np.ndarray] = None

    def _c(self):
        A = _operand(self.A, self.a_type)
        B = _operand(self.B, self.b_type)
        M, K = A.shape
        N = B.shape[0] if self.b_is_nk else B.shape[1]
        B2 = _operand(self.B2, self.b_type)
        if B2 is not None:
            if B2.shape != B.shape:
                raise ValueError("B2 must have B's shape")
            N *= 2
        if (B.shape[1] if self.b_is_nk else B.shape[0]) != K:
            raise ValueError("A and B disagree on K")
        keep = [A, B, B2]
        bias = _f32(self.bias)
        rs = _f32(self.row_scale)
        res = _u16(self.residual)
        pre = _u16(self.preact)
        cs = _f32(self.col_scale)
        keep += [bias, rs, res, pre, cs]
        aux = res if res is not None else pre
        ld_aux = aux.shape[1] if aux is not None else 0
        prog = ",".join(self.program).encode()
        keep.append(prog)
        p = _Problem(M, N, K, 1 if self.b_is_nk else 0,
                     A.ctypes.data, A.shape[1], B.ctypes.data, B.shape[1], _ptr(B2),
                     float(self.alpha), _ptr(bias), _ptr(rs), _ptr(res), _ptr(pre),
                     ld_aux, float(self.fp8_scale), prog, TYPES[self.a_type], TYPES[self.b_type],
                     float(self.a_scale_inv), float(self.b_scale_inv), _ptr(cs))
        return p, keep

    @property
    def M(self):
        return self.A.shape[0]

    def out_cols(self) -> int:
        p, keep = self._c()
        n = load().oracle_out_cols(ctypes.byref(p))
        if n < 0:
            raise ValueError("bad program %r" % (self.program,))
        return n

    def rows(self, rows: Optional[Sequence[int]] = None) -> dict:
        """Whole output rows.  Returns y (fp64 value at the bf16 store),
        c_bf16 (uint16 bits), c_e4m3 (uint8 codes), row_stat and amax_rows."""
        p, keep = self._c()
        lib = load()
        nout = self.out_cols()
        if rows is None:
            idx = None
            nrows = self.M
        else:
            idx = np.ascontiguousarray(rows, dtype=np.int64)
            nrows = idx.shape[0]
        y = np.empty((nrows, nout), np.float64)
        cb = np.empty((nrows, nout), np.uint16)
        c8 = np.empty((nrows, nout), np.uint8)
        rs = np.empty(nrows, np.float64)
        am = np.empty(nrows, np.float64)
        rc = lib.oracle_rows(ctypes.byref(p), _ptr(idx), nrows, _ptr(y), _ptr(cb), _ptr(c8),
                             _ptr(rs), _ptr(am))
        if rc != 0:
            raise ValueError("oracle_rows failed (%d)" % rc)
        return {"y": y, "c_bf16": cb, "c_e4m3": c8, "row_stat": rs, "amax_rows": am,
                "amax": float(am.max()) if nrows else 0.0}

    def cols(self, cols: Sequence[int]) -> dict:
        """Whole output columns (all M rows): y (M x ncols) and col_stat."""
        p, keep = self._c()
        lib = load()
        idx = np.ascontiguousarray(cols, dtype=np.int64)
        y = np.empty((self.M, idx.shape[0]), np.float64)
        cs = np.empty(idx.shape[0], np.float64)
        rc = lib.oracle_cols(ctypes.byref(p), _ptr(idx), idx.shape[0], _ptr(y), _ptr(cs))
        if rc != 0:
            raise ValueError("oracle_cols failed (%d)" % rc)
        return {"y": y, "col_stat": cs}


def rmsnorm_backward(dy, x, s, r, w=None, add=None, want_dx=True, want_dw=True):
    """RMSNorm backward from the row reduction r (see oracle.h): returns
    (dx, dw) in fp64; dy, x, add are bf16 bit patterns (uint16)."""
    dy, x, add = _u16(dy), _u16(x), _u16(add)
    M, N = dy.shape
    s = _f32(s)
    r = np.ascontiguousarray(r, dtype=np.float64)
    w = _f32(w)
    dx = np.empty((M, N), np.float64) if want_dx else None
    dw = np.empty(N, np.float64) if want_dw else None
    load().oracle_rmsnorm_backward(M, N, _ptr(dy), dy.shape[1], _ptr(x), x.shape[1], _ptr(w), _ptr(s), _ptr(r),
                                   _ptr(add), 0 if add is None else add.shape[1], _ptr(dx), _ptr(dw))
    return dx, dw


def gelu_tanh(x: float) -> float:
    return load().oracle_gelu_tanh(x)


def gelu_tanh_grad(x: float) -> float:
    return load().oracle_gelu_tanh_grad(x)


def silu(x: float) -> float:
    return load().oracle_silu(x)


def silu_grad(x: float) -> float:
    return load().oracle_silu_grad(x)


def to_bf16_bits(x) -> np.ndarray:
    f = load().oracle_double_to_bf16
    a = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


def bf16_bits_to_f64(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_e4m3(x) -> np.ndarray:
    f = load().oracle_double_to_e4m3
    a = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def e4m3_to_f64(c) -> np.ndarray:
    f = load().oracle_e4m3_to_double
    a = np.asarray(c, dtype=np.uint8)
    return np.array([f(int(v)) for v in a.ravel()], dtype=np.float64).reshape(a.shape)


def e5m2_to_f64(c) -> np.ndarray:
    f = load().oracle_e5m2_to_double
    a = np.asarray(c, dtype=np.uint8)
    return np.array([f(int(v)) for v in a.ravel()], dtype=np.float64).reshape(a.shape)


def cpu_threads() -> int:
    """Threads the oracle's OpenMP loops use in this process."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env:
        return int(env)
    return len(os.sched_getaffinity(0))
