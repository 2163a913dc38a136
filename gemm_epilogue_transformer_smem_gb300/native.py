"""ctypes binding of the C ABI in include/gemm_epi.h (same names, argument
marshalling only).  Loading fails loudly when the built library is missing:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libgemm_epi.so")

# gemm_epi_status
GEMM_EPI_OK = 0
GEMM_EPI_ERR_INVALID_VALUE = 1
GEMM_EPI_ERR_MISALIGNED = 2
GEMM_EPI_ERR_UNSUPPORTED = 3
GEMM_EPI_ERR_ARCH = 4
GEMM_EPI_ERR_CUDA = 5
GEMM_EPI_ERR_TIMEOUT = 6
GEMM_EPI_ERR_WORKSPACE = 7

STATUS_NAMES = {
    0: "GEMM_EPI_OK", 1: "GEMM_EPI_ERR_INVALID_VALUE", 2: "GEMM_EPI_ERR_MISALIGNED",
    3: "GEMM_EPI_ERR_UNSUPPORTED", 4: "GEMM_EPI_ERR_ARCH", 5: "GEMM_EPI_ERR_CUDA",
    6: "GEMM_EPI_ERR_TIMEOUT", 7: "GEMM_EPI_ERR_WORKSPACE",
}

# gemm_epi_type
GEMM_EPI_TYPE_BF16 = 0
GEMM_EPI_TYPE_E4M3 = 1
GEMM_EPI_TYPE_E5M2 = 2

# gemm_epi_b_layout
GEMM_EPI_B_KN = 0
GEMM_EPI_B_NK = 1
GEMM_EPI_B_DUAL = 16

# gemm_epi_op_code
GEMM_EPI_OP_SCALE_ALPHA = 1
GEMM_EPI_OP_ADD_BIAS_COL = 2
GEMM_EPI_OP_MUL_ROW_SCALE = 3
GEMM_EPI_OP_ADD_RESIDUAL = 4
GEMM_EPI_OP_ACT_GELU_TANH = 5
GEMM_EPI_OP_ACT_RELU = 6
GEMM_EPI_OP_ACT_SILU = 7
GEMM_EPI_OP_PAIR_SWIGLU = 8
GEMM_EPI_OP_MUL_GELU_TANH_GRAD = 9
GEMM_EPI_OP_AMAX = 10
GEMM_EPI_OP_STORE_BF16 = 11
GEMM_EPI_OP_STORE_E4M3 = 12
GEMM_EPI_OP_ROW_RMS_RSQRT = 13
GEMM_EPI_OP_COL_SUM = 14
GEMM_EPI_OP_PAIR_MUL = 15
GEMM_EPI_OP_DSWIGLU = 16
GEMM_EPI_OP_MUL_COL_SCALE = 17
GEMM_EPI_OP_ROW_DOT = 18

GEMM_EPI_MAX_OPS = 16
GEMM_EPI_DEBUG_SKIP_FIRST_LOAD = 1
GEMM_EPI_DEBUG_FORCE_1SM = 2
GEMM_EPI_DEBUG_FORCE_2SM = 4
GEMM_EPI_DEBUG_FORCE_INTERPRETER = 8
GEMM_EPI_DEBUG_SKIP_SECOND_LOAD = 16
GEMM_EPI_NO_ALLOC_SCRATCH_BYTES = 65536


class gemm_epi_op(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int32), ("i0", ctypes.c_int32), ("f0", ctypes.c_float)]


class gemm_epi_desc(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64),
        ("ldc", ctypes.c_int64), ("ldc8", ctypes.c_int64), ("ld_aux", ctypes.c_int64),
        ("b_layout", ctypes.c_int32), ("n_ops", ctypes.c_int32),
        ("ops", ctypes.POINTER(gemm_epi_op)),
        ("batch", ctypes.c_int64),
        ("batch_stride_a", ctypes.c_int64), ("batch_stride_b", ctypes.c_int64),
        ("batch_stride_c", ctypes.c_int64), ("batch_stride_c8", ctypes.c_int64),
        ("batch_stride_aux", ctypes.c_int64),
        ("a_type", ctypes.c_int32), ("b_type", ctypes.c_int32),
    ]


class gemm_epi_args(ctypes.Structure):
    _fields_ = [
        ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
        ("alpha", ctypes.c_float), ("fp8_scale", ctypes.c_float),
        ("bias", ctypes.c_void_p), ("row_scale", ctypes.c_void_p),
        ("residual", ctypes.c_void_p), ("preact", ctypes.c_void_p),
        ("C", ctypes.c_void_p), ("C8", ctypes.c_void_p),
        ("amax", ctypes.c_void_p), ("row_out", ctypes.c_void_p), ("col_out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("timeout_ms", ctypes.c_uint32), ("debug_flags", ctypes.c_uint32),
        ("B2", ctypes.c_void_p),
        ("a_scale_inv", ctypes.c_void_p), ("b_scale_inv", ctypes.c_void_p),
        ("col_scale", ctypes.c_void_p),
    ]


class gemm_epi_rmsnorm_bwd_args(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64),
        ("dy", ctypes.c_void_p), ("ld_dy", ctypes.c_int64),
        ("x", ctypes.c_void_p), ("ld_x", ctypes.c_int64),
        ("add", ctypes.c_void_p), ("ld_add", ctypes.c_int64),
        ("w", ctypes.c_void_p), ("s", ctypes.c_void_p), ("r", ctypes.c_void_p),
        ("dx", ctypes.c_void_p), ("ld_dx", ctypes.c_int64),
        ("dw", ctypes.c_void_p),
    ]


gemm_epi_handle = ctypes.c_void_p

# (name, restype, argtypes): every entry point declared in include/gemm_epi.h.
SIGNATURES = [
    ("gemm_epi_create", ctypes.c_int, [ctypes.POINTER(gemm_epi_handle), ctypes.POINTER(gemm_epi_desc)]),
    ("gemm_epi_destroy", ctypes.c_int, [gemm_epi_handle]),
    ("gemm_epi_workspace_size", ctypes.c_size_t, [gemm_epi_handle]),
    ("gemm_epi_out_cols", ctypes.c_int64, [gemm_epi_handle]),
    ("gemm_epi_run", ctypes.c_int, [gemm_epi_handle, ctypes.POINTER(gemm_epi_args), ctypes.c_void_p]),
    ("gemm_epi_run_unfused", ctypes.c_int,
     [gemm_epi_handle, ctypes.POINTER(gemm_epi_args), ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
    ("gemm_epi_run_no_alloc", ctypes.c_int, [gemm_epi_handle, ctypes.POINTER(gemm_epi_args), ctypes.c_void_p]),
    ("gemm_epi_rmsnorm_backward", ctypes.c_int, [ctypes.POINTER(gemm_epi_rmsnorm_bwd_args), ctypes.c_void_p]),
    ("gemm_epi_query_status", ctypes.c_int, [gemm_epi_handle, ctypes.c_void_p, ctypes.c_void_p]),
    ("gemm_epi_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("gemm_epi_last_error", ctypes.c_char_p, []),
    ("gemm_epi_version", ctypes.c_int, []),
]

_lib = None


def load(path: str = LIB_PATH):
    """Loads the built library (build it with ``build.build()``)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            "CUDA library %s is missing; build it with "
            "gemm_epilogue_transformer_smem_gb300.build.build()" % path)
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


class GemmEpiError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, str(status)), message))


def check(status: int, lib=None):
    if status != GEMM_EPI_OK:
        lib = lib or load()
        raise GemmEpiError(status, lib.gemm_epi_last_error().decode(errors="replace"))
    return status
