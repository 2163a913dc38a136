"""Torch-facing wrapper over the C ABI: builds the descriptor from an op list,
passes tensor data pointers and the current CUDA stream.  No arithmetic of the
method happens here; every step runs in the CUDA library.

Programs are written as op names (one optional numeric argument after a
colon):

  alpha, bias, row_scale, residual, gelu_tanh, relu, silu, pair_swiglu[:g], pair_mul[:g],
  gelu_tanh_grad, amax, store_bf16, store_e4m3, row_rms[:eps],
  row_rms_unrounded[:eps], col_sum, dswiglu[:g], col_scale, row_dot
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import native as N

PROGRAM_OPS = {
    "alpha": N.GEMM_EPI_OP_SCALE_ALPHA,
    "bias": N.GEMM_EPI_OP_ADD_BIAS_COL,
    "row_scale": N.GEMM_EPI_OP_MUL_ROW_SCALE,
    "residual": N.GEMM_EPI_OP_ADD_RESIDUAL,
    "gelu_tanh": N.GEMM_EPI_OP_ACT_GELU_TANH,
    "relu": N.GEMM_EPI_OP_ACT_RELU,
    "silu": N.GEMM_EPI_OP_ACT_SILU,
    "pair_swiglu": N.GEMM_EPI_OP_PAIR_SWIGLU,
    "pair_mul": N.GEMM_EPI_OP_PAIR_MUL,
    "dswiglu": N.GEMM_EPI_OP_DSWIGLU,
    "col_scale": N.GEMM_EPI_OP_MUL_COL_SCALE,
    "row_dot": N.GEMM_EPI_OP_ROW_DOT,
    "gelu_tanh_grad": N.GEMM_EPI_OP_MUL_GELU_TANH_GRAD,
    "amax": N.GEMM_EPI_OP_AMAX,
    "store_bf16": N.GEMM_EPI_OP_STORE_BF16,
    "store_e4m3": N.GEMM_EPI_OP_STORE_E4M3,
    "row_rms": N.GEMM_EPI_OP_ROW_RMS_RSQRT,
    "row_rms_unrounded": N.GEMM_EPI_OP_ROW_RMS_RSQRT,
    "col_sum": N.GEMM_EPI_OP_COL_SUM,
}


def encode_program(program: Sequence[str]):
    ops = (N.gemm_epi_op * max(1, len(program)))()
    for i, spec in enumerate(program):
        name, _, arg = spec.partition(":")
        if name not in PROGRAM_OPS:
            raise ValueError("unknown epilogue op %r" % name)
        code = PROGRAM_OPS[name]
        i0, f0 = 0, 0.0
        if name in ("pair_swiglu", "pair_mul", "dswiglu"):
            i0 = int(arg) if arg else 1
        elif name.startswith("row_rms"):
            f0 = float(arg) if arg else 1e-6
            i0 = 1 if name == "row_rms_unrounded" else 0
        ops[i] = N.gemm_epi_op(code, i0, f0)
    return ops


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _bytes_after(t: torch.Tensor) -> int:
    """Bytes of the tensor's storage from its first element to the end."""
    return t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()


def _expect(name: str, t: Optional[torch.Tensor], kind: str, rows: int, cols: int = 1, ld: int = 1,
            batch: int = 1, batch_stride: int = 0) -> None:
    """Checks one buffer before its pointer crosses the C ABI, which sees
    neither dtype nor size: ``kind`` is "bf16", "f32" or "byte" (any 8-bit
    type), and the storage must hold ``batch`` matrices of ``rows`` x ``cols``
    elements at row stride ``ld`` and batch stride ``batch_stride``."""
    if t is None:
        return
    ok = {"bf16": t.dtype == torch.bfloat16, "f32": t.dtype == torch.float32,
          "byte": t.element_size() == 1}[kind]
    if not ok:
        raise TypeError("%s: expected a %s tensor, got %s" % (name, kind, t.dtype))
    if batch <= 0 or rows <= 0 or cols <= 0:
        return
    need = ((batch - 1) * batch_stride + (rows - 1) * ld + cols) * t.element_size()
    if need > _bytes_after(t):
        raise ValueError("%s: %d bytes needed from its first element, the storage holds %d"
                         % (name, need, _bytes_after(t)))


def _width_at(program: Sequence[str], N_: int):
    """Accumulator width each op sees: N before a pair op, N/2 after it, 2N
    after dswiglu."""
    w, out = N_, []
    for spec in program:
        name = spec.partition(":")[0]
        out.append((name, w))
        if name.startswith("pair_"):
            w = N_ // 2
        elif name == "dswiglu":
            w = 2 * N_
    return out


# Operand element types (desc.a_type / b_type); 8-bit operands are passed as
# uint8 (or torch float8) tensors of codes.
OPERAND_TYPES = {"bf16": N.GEMM_EPI_TYPE_BF16, "e4m3": N.GEMM_EPI_TYPE_E4M3, "e5m2": N.GEMM_EPI_TYPE_E5M2}


# Ops that read the auxiliary M x N_out tensor, by the argument it travels in.
RESIDUAL_OPS = frozenset({"residual", "row_dot"})
PREACT_OPS = frozenset({"gelu_tanh_grad", "dswiglu"})


def out_cols(program: Sequence[str], N_: int) -> int:
    """Output columns of a program over N accumulator columns."""
    names = [op.partition(":")[0] for op in program]
    if "dswiglu" in names:
        return 2 * N_
    return N_ // 2 if any(n.startswith("pair_") for n in names) else N_


class Plan:
    """One validated GEMM + epilogue plan (gemm_epi_create).  Strides default
    to tight row-major packing."""

    def __init__(self, M: int, N_: int, K: int, program: Sequence[str], b_layout: str = "kn",
                 lda: Optional[int] = None, ldb: Optional[int] = None, ldc: Optional[int] = None,
                 ldc8: Optional[int] = None, ld_aux: Optional[int] = None, dual: bool = False,
                 batch: int = 1, batch_stride_a: Optional[int] = None,
                 batch_stride_b: Optional[int] = None, batch_stride_c: Optional[int] = None,
                 batch_stride_c8: Optional[int] = None, batch_stride_aux: Optional[int] = None,
                 a_type: str = "bf16", b_type: str = "bf16"):
        self.lib = N.load()
        self.program = list(program)
        self.M, self.N, self.K = M, N_, K
        self.b_layout = b_layout
        n_out = out_cols(program, N_)
        self._ops = encode_program(program)
        d = N.gemm_epi_desc()
        d.M, d.N, d.K = M, N_, K
        d.lda = K if lda is None else lda
        b_cols = N_ // 2 if dual else N_
        d.ldb = (b_cols if b_layout == "kn" else K) if ldb is None else ldb
        d.ldc = n_out if ldc is None else ldc
        d.ldc8 = n_out if ldc8 is None else ldc8
        d.ld_aux = n_out if ld_aux is None else ld_aux
        d.b_layout = (N.GEMM_EPI_B_KN if b_layout == "kn" else N.GEMM_EPI_B_NK) | (N.GEMM_EPI_B_DUAL if dual else 0)
        self.dual = dual
        d.n_ops = len(program)
        d.ops = ctypes.cast(self._ops, ctypes.POINTER(N.gemm_epi_op))
        # Batched: tight packing by default; a stride of 0 shares A or B.
        d.batch = batch
        b_rows = K if b_layout == "kn" else b_cols
        d.batch_stride_a = M * d.lda if batch_stride_a is None else batch_stride_a
        d.batch_stride_b = b_rows * d.ldb if batch_stride_b is None else batch_stride_b
        d.batch_stride_c = M * d.ldc if batch_stride_c is None else batch_stride_c
        d.batch_stride_c8 = M * d.ldc8 if batch_stride_c8 is None else batch_stride_c8
        d.batch_stride_aux = M * d.ld_aux if batch_stride_aux is None else batch_stride_aux
        self.batch = batch
        d.a_type, d.b_type = OPERAND_TYPES[a_type], OPERAND_TYPES[b_type]
        self.a_type, self.b_type = a_type, b_type
        self.desc = d
        h = N.gemm_epi_handle()
        N.check(self.lib.gemm_epi_create(ctypes.byref(h), ctypes.byref(d)), self.lib)
        self.handle = h
        self.n_out = int(self.lib.gemm_epi_out_cols(h))
        self.workspace_bytes = int(self.lib.gemm_epi_workspace_size(h))

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            self.lib.gemm_epi_destroy(h)
            self.handle = None

    def args(self, A, B, *, alpha=1.0, fp8_scale=1.0, bias=None, row_scale=None, residual=None,
             preact=None, C=None, C8=None, amax=None, row_out=None, col_out=None, workspace=None,
             timeout_ms=0, debug_flags=0, B2=None, a_scale_inv=None, b_scale_inv=None,
             col_scale=None) -> N.gemm_epi_args:
        a = N.gemm_epi_args()
        a.A, a.B, a.B2 = _ptr(A), _ptr(B), _ptr(B2)
        a.a_scale_inv, a.b_scale_inv = _ptr(a_scale_inv), _ptr(b_scale_inv)
        a.col_scale = _ptr(col_scale)
        a.alpha, a.fp8_scale = float(alpha), float(fp8_scale)
        a.bias, a.row_scale = _ptr(bias), _ptr(row_scale)
        a.residual, a.preact = _ptr(residual), _ptr(preact)
        a.C, a.C8 = _ptr(C), _ptr(C8)
        a.amax, a.row_out, a.col_out = _ptr(amax), _ptr(row_out), _ptr(col_out)
        a.workspace = _ptr(workspace)
        a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        a.timeout_ms, a.debug_flags = int(timeout_ms), int(debug_flags)
        self._check(A, B, B2, bias, row_scale, residual, preact, C, C8, amax, row_out, col_out,
                    a_scale_inv, b_scale_inv, col_scale)
        return a

    def _check(self, A, B, B2, bias, row_scale, residual, preact, C, C8, amax, row_out, col_out,
               a_scale_inv, b_scale_inv, col_scale):
        d, M, K, Bt = self.desc, self.M, self.K, self.batch
        op_kind = lambda t: "bf16" if t == "bf16" else "byte"  # noqa: E731
        b_cols = self.N // 2 if self.dual else self.N
        b_rows, b_inner = (K, b_cols) if self.b_layout == "kn" else (b_cols, K)
        _expect("A", A, op_kind(self.a_type), M, K, d.lda, Bt, d.batch_stride_a)
        _expect("B", B, op_kind(self.b_type), b_rows, b_inner, d.ldb, Bt, d.batch_stride_b)
        _expect("B2", B2, op_kind(self.b_type), b_rows, b_inner, d.ldb, Bt, d.batch_stride_b)
        _expect("C", C, "bf16", M, self.n_out, d.ldc, Bt, d.batch_stride_c)
        _expect("C8", C8, "byte", M, self.n_out, d.ldc8, Bt, d.batch_stride_c8)
        for name, t in (("residual", residual), ("preact", preact)):
            _expect(name, t, "bf16", M, self.n_out, d.ld_aux, Bt, d.batch_stride_aux)
        _expect("row_scale", row_scale, "f32", Bt * M)
        _expect("row_out", row_out, "f32", Bt * M)
        _expect("col_out", col_out, "f32", Bt * self.n_out)
        for name, t in (("amax", amax), ("a_scale_inv", a_scale_inv), ("b_scale_inv", b_scale_inv)):
            _expect(name, t, "f32", 1)
        widths = dict((op, w) for op, w in _width_at(self.program, self.N))
        _expect("bias", bias, "f32", widths.get("bias", 1))
        _expect("col_scale", col_scale, "f32", widths.get("col_scale", 1))

    def run(self, *tensors, stream: Optional[torch.cuda.Stream] = None, **kw):
        """gemm_epi_run on the current (or given) CUDA stream; asynchronous."""
        a = self.args(*tensors, **kw)
        s = (stream or torch.cuda.current_stream()).cuda_stream
        N.check(self.lib.gemm_epi_run(self.handle, ctypes.byref(a), ctypes.c_void_p(s)), self.lib)

    def run_unfused(self, *tensors, scratch: torch.Tensor, stream=None, **kw):
        a = self.args(*tensors, **kw)
        _expect("scratch", scratch, "bf16", self.M, self.N, scratch.stride(0))
        s = (stream or torch.cuda.current_stream()).cuda_stream
        N.check(self.lib.gemm_epi_run_unfused(self.handle, ctypes.byref(a), ctypes.c_void_p(scratch.data_ptr()),
                                              scratch.stride(0), ctypes.c_void_p(s)), self.lib)

    def query_status(self, workspace: torch.Tensor, stream=None) -> int:
        s = (stream or torch.cuda.current_stream()).cuda_stream
        return int(self.lib.gemm_epi_query_status(self.handle, ctypes.c_void_p(workspace.data_ptr()),
                                                  ctypes.c_void_p(s)))


@dataclass
class Outputs:
    C: Optional[torch.Tensor] = None
    C8: Optional[torch.Tensor] = None
    amax: Optional[torch.Tensor] = None
    row_out: Optional[torch.Tensor] = None
    col_out: Optional[torch.Tensor] = None
    workspace: Optional[torch.Tensor] = None


def allocate_outputs(plan: Plan, device) -> Outputs:
    """Device buffers for every output the program writes (torch allocates)."""
    prog = [op.partition(":")[0] for op in plan.program]
    o = Outputs()
    lead = (plan.batch,) if plan.batch > 1 else ()
    if "store_bf16" in prog:
        o.C = torch.empty(lead + (plan.M, plan.n_out), dtype=torch.bfloat16, device=device)
    if "store_e4m3" in prog:
        o.C8 = torch.empty(lead + (plan.M, plan.n_out), dtype=torch.uint8, device=device)
    if "amax" in prog:
        o.amax = torch.empty(1, dtype=torch.float32, device=device)
    if any(p.startswith("row_rms") or p == "row_dot" for p in prog):
        o.row_out = torch.empty(lead + (plan.M,), dtype=torch.float32, device=device)
    if "col_sum" in prog:
        o.col_out = torch.empty(lead + (plan.n_out,), dtype=torch.float32, device=device)
    o.workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=device)
    return o


def run_program(plan: Plan, A, B, out: Outputs, *, alpha=1.0, fp8_scale=1.0, bias=None,
                row_scale=None, aux=None, unfused_scratch=None, **kw) -> Outputs:
    """Runs the plan with the auxiliary tensor routed to residual or preact."""
    prog = [op.partition(":")[0] for op in plan.program]
    residual = aux if any(op in RESIDUAL_OPS for op in prog) else None
    preact = aux if any(op in PREACT_OPS for op in prog) else None
    tensors = dict(alpha=alpha, fp8_scale=fp8_scale, bias=bias, row_scale=row_scale,
                   residual=residual, preact=preact, C=out.C, C8=out.C8, amax=out.amax,
                   row_out=out.row_out, col_out=out.col_out, workspace=out.workspace, **kw)
    if unfused_scratch is not None:
        plan.run_unfused(A, B, scratch=unfused_scratch, **tensors)
    else:
        plan.run(A, B, **tensors)
    return out


def rmsnorm_backward(dy, x, s, r, *, w=None, add=None, dx=None, dw=None, stream=None):
    """gemm_epi_rmsnorm_backward: dx = S w dy - x S^3 r / N (+ add) into `dx`
    and dw = sum_m dy x S into `dw` (either may be None); bf16 2-D tensors
    with unit column stride, fp32 vectors.  Asynchronous."""
    lib = N.load()
    a = N.gemm_epi_rmsnorm_bwd_args()
    a.M, a.N = dy.shape
    for name, t in (("dy", dy), ("x", x), ("add", add), ("dx", dx)):
        _expect(name, t, "bf16", a.M, a.N, 1 if t is None else t.stride(0))
    for name, t, n in (("s", s, a.M), ("r", r, a.M), ("w", w, a.N), ("dw", dw, a.N)):
        _expect(name, t, "f32", n)
    a.dy, a.ld_dy = _ptr(dy), dy.stride(0)
    a.x, a.ld_x = _ptr(x), x.stride(0)
    a.add, a.ld_add = _ptr(add), (add.stride(0) if add is not None else 0)
    a.w, a.s, a.r = _ptr(w), _ptr(s), _ptr(r)
    a.dx, a.ld_dx = _ptr(dx), (dx.stride(0) if dx is not None else 0)
    a.dw = _ptr(dw)
    st = (stream or torch.cuda.current_stream()).cuda_stream
    N.check(lib.gemm_epi_rmsnorm_backward(ctypes.byref(a), ctypes.c_void_p(st)), lib)
