"""Seeded synthetic inputs for the GEMM + epilogue workloads.

This module holds shapes, value distributions and random draws only -- none
of the method's arithmetic.  Both the CUDA path and the CPU oracle read the
tensors it returns (the oracle through host copies of the same bf16 bits).

Workloads (shapes and distributions as the benchmark configuration states
them; "N(0, s)" has standard deviation s):

  tiny      C = gelu_tanh(1.0 * A@B + bias), AMAX.  A 64x128, B 128x64, both
            N(0,1)/sqrt(128); bias fp32 N(0, 0.1), length 64.
  swiglu    MLP up-projection, out = silu(gate) * up on interleaved columns.
            A 8192x4096 N(0,1); B 4096x28672 N(0, 0.02).
  fp8       relu(0.5 * A@B + bias), AMAX, bf16 C and e4m3 C with scale 448/4.
            M = N = K = 8192, A and B N(0,1)/sqrt(8192); bias N(0, 0.1).
  downproj  out = residual + A@B, per-row rsqrt(mean(out^2) + 1e-6).
            A 16384x14336 N(0,1)/sqrt(14336); B 14336x4096 N(0, 0.02);
            residual 16384x4096 N(0,1).
  swiglu2w  the same up-projection with separate gate and up weights:
            out = silu(A @ W_gate) * (A @ W_up), W_gate and W_up 4096x14336 each
            N(0, 0.02).
  backward  dX = (dY @ W^T) * gelu_tanh'(preact), column sums of dX.
            dY 8192x4096 N(0,1); W 16384x4096 N(0, 0.02); preact 8192x16384
            N(0,1).
  dswiglu   the SwiGLU backward of the swiglu workload's MLP: dH = dY @ W_down^T
            with the gradients of both gate and up written from dH and the
            forward pre-activations.  dY 8192x4096 N(0,1); W_down stored
            14336x4096 (N x K) N(0, 0.02); preact (the forward gate / up pairs,
            interleaved) 8192x28672 N(0, 1.28), the spread of the swiglu
            workload's own GEMM output (0.02 * sqrt(4096)); out 8192x28672.
  drmsnorm  the RMSNorm backward at the down-projection's output: dy = dH @ W
            (dH 16384x14336 N(0,1), W 14336x4096 N(0, 0.02)) is stored, scaled
            by the norm weight w (fp32 N(1, 0.1)) and reduced against the
            RMSNorm input x (the residual stream, 16384x4096 N(0,1)) per row;
            a second pass (gemm_epi_rmsnorm_backward) gives dx and dw from it
            and the forward's S (fp32, 1 + N(0, 0.05), what the forward's row
            statistic holds for rows of unit mean square).
  fp8in     the fp8 workload's program on FP8 operands: the next layer of the
            FP8 loop reads the e4m3 activations the fp8 workload emits.
            M = N = K = 8192.  A: e4m3 codes of max(N(0, 0.1), 0) * 112 (the
            fp8 workload's output distribution, its bias dominating, at its
            scale 448/4), dequantised by 1/112.  B: a weight stored N x K,
            N(0,1)/sqrt(K), as e4m3 codes at scale 112 * sqrt(K) (448/4 of its
            own standard deviation), dequantised by the reciprocal.
  rmsswiglu the RMSNorm-consuming up-projection: the swiglu workload's GEMM
            with its rows scaled by the previous layer's S before the pair
            op, out = silu(S*gate) * (S*up).  A (the unnormalised residual
            stream) 8192x4096 N(0,1); B 4096x28672 N(0, 0.02); S fp32
            1 + N(0, 0.05) per row.
  rmsglu    the same with the RMSNorm-MLP's plain product, out = (S*gate) *
            (S*up).
  moe8      eight independent SwiGLU up-projections in one launch (one per
            expert, each with its own weights): per expert A 2048x4096
            N(0,1), B 4096x28672 N(0, 0.02).
  decode    the swiglu workload's up-projection for one decode step of 64
            tokens: A 64x4096 N(0,1), B 4096x28672 N(0, 0.02).  Reading B
            dominates, so the HBM roofline binds.

Draw order per workload: A, B, bias, residual / preact, B2, column scale, S,
row scale.  A batched workload draws each tensor for every batch at once.  Each tensor is drawn
in fp32 with ``torch.randn`` from one generator seeded with 1000 + index,
scaled, then cast to bf16 (round to nearest even); bias stays fp32.  FP8
operands are multiplied by their quantisation scale, clamped to the format's
largest finite value and cast with torch (round to nearest even); the
reciprocal scales travel as one-element fp32 device tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    M: int
    N: int               # accumulator columns (B's N)
    K: int
    b_layout: str        # "kn": B stored K x N; "nk": B stored N x K (B = W^T)
    program: tuple       # op names, oracle spelling; see api.PROGRAM_OPS
    a_std: float
    b_std: float
    bias_std: Optional[float] = None
    aux: Optional[str] = None       # "residual" or "preact"
    aux_std: float = 1.0
    alpha: float = 1.0
    fp8_scale: float = 1.0
    dual: bool = False   # B holds gate columns, B2 the matching up columns (N/2 each)
    in_type: str = "bf16"   # operand type of A and B: "bf16" or "e4m3"
    a_relu: bool = False    # A drawn as max(N(0, a_std), 0)
    a_qscale: float = 1.0   # FP8 quantisation scales of A and B
    b_qscale: float = 1.0
    col_scale_std: Optional[float] = None   # column scale drawn as 1 + N(0, std)
    finish: Optional[str] = None            # a second pass after the GEMM ("rmsnorm_backward")
    row_scale_std: Optional[float] = None   # row scale (the consumed S) drawn as 1 + N(0, std)
    batch: int = 1                          # independent problems of this shape in one launch
    notes: str = ""

    @property
    def n_out(self) -> int:
        names = [op.partition(":")[0] for op in self.program]
        if "dswiglu" in names:
            return 2 * self.N
        return self.N // 2 if any(n.startswith("pair_") for n in names) else self.N

    @property
    def flops(self) -> int:
        return 2 * self.batch * self.M * self.N * self.K

    def scaled(self, M: int, N: int, K: int, name: Optional[str] = None) -> "Workload":
        """Same program and distributions at another shape.  Standard
        deviations that the full workload ties to K (1/sqrt(K)) follow K."""
        a_std, b_std = self.a_std, self.b_std
        if self.name in ("tiny", "fp8", "downproj"):
            a_std = 1.0 / math.sqrt(K)
        if self.name in ("tiny", "fp8", "fp8in"):
            b_std = 1.0 / math.sqrt(K)
        b_qscale = 112.0 * math.sqrt(K) if self.name == "fp8in" else self.b_qscale
        return replace(self, name=name or "%s_%dx%dx%d" % (self.name, M, N, K), M=M, N=N, K=K,
                       a_std=a_std, b_std=b_std, b_qscale=b_qscale)


WORKLOADS = {
    "tiny": Workload("tiny", 0, 64, 64, 128, "kn",
                     ("alpha", "bias", "gelu_tanh", "amax", "store_bf16"),
                     a_std=1 / math.sqrt(128), b_std=1 / math.sqrt(128), bias_std=0.1,
                     alpha=1.0),
    "swiglu": Workload("swiglu", 1, 8192, 28672, 4096, "kn",
                       ("pair_swiglu", "store_bf16"),
                       a_std=1.0, b_std=0.02),
    "fp8": Workload("fp8", 2, 8192, 8192, 8192, "kn",
                    ("alpha", "bias", "relu", "amax", "store_bf16", "store_e4m3"),
                    a_std=1 / math.sqrt(8192), b_std=1 / math.sqrt(8192), bias_std=0.1,
                    alpha=0.5, fp8_scale=448.0 / 4.0),
    "downproj": Workload("downproj", 3, 16384, 4096, 14336, "kn",
                         ("residual", "store_bf16", "row_rms:1e-6"),
                         a_std=1 / math.sqrt(14336), b_std=0.02, aux="residual"),
    "swiglu2w": Workload("swiglu2w", 5, 8192, 28672, 4096, "kn",
                         ("pair_swiglu:128", "store_bf16"),
                         a_std=1.0, b_std=0.02, dual=True),
    "backward": Workload("backward", 4, 8192, 16384, 4096, "nk",
                         ("gelu_tanh_grad", "store_bf16", "col_sum"),
                         a_std=1.0, b_std=0.02, aux="preact"),
    "dswiglu": Workload("dswiglu", 7, 8192, 14336, 4096, "nk", ("dswiglu", "store_bf16"),
                        a_std=1.0, b_std=0.02, aux="preact", aux_std=1.28),
    "drmsnorm": Workload("drmsnorm", 8, 16384, 4096, 14336, "kn", ("store_bf16", "col_scale", "row_dot"),
                         a_std=1.0, b_std=0.02, aux="residual", col_scale_std=0.1,
                         finish="rmsnorm_backward"),
    "fp8in": Workload("fp8in", 6, 8192, 8192, 8192, "nk",
                      ("alpha", "bias", "relu", "amax", "store_bf16", "store_e4m3"),
                      a_std=0.1, b_std=1 / math.sqrt(8192), bias_std=0.1, alpha=0.5,
                      fp8_scale=448.0 / 4.0, in_type="e4m3", a_relu=True, a_qscale=112.0,
                      b_qscale=112.0 * math.sqrt(8192)),
    "rmsswiglu": Workload("rmsswiglu", 9, 8192, 28672, 4096, "kn", ("row_scale", "pair_swiglu", "store_bf16"),
                          a_std=1.0, b_std=0.02, row_scale_std=0.05),
    "rmsglu": Workload("rmsglu", 10, 8192, 28672, 4096, "kn", ("row_scale", "pair_mul", "store_bf16"),
                       a_std=1.0, b_std=0.02, row_scale_std=0.05),
    "moe8": Workload("moe8", 11, 2048, 28672, 4096, "kn", ("pair_swiglu", "store_bf16"),
                     a_std=1.0, b_std=0.02, batch=8),
    "decode": Workload("decode", 12, 64, 28672, 4096, "kn", ("pair_swiglu", "store_bf16"),
                       a_std=1.0, b_std=0.02),
}

BY_INDEX = {w.index: w for w in WORKLOADS.values()}


@dataclass
class Inputs:
    A: torch.Tensor                 # M x K bf16
    B: torch.Tensor                 # K x N or N x K bf16 (N/2 columns with a B2)
    bias: Optional[torch.Tensor]    # fp32, length = columns where the bias op sits
    aux: Optional[torch.Tensor]     # M x n_out bf16 (residual or preact)
    alpha: float
    fp8_scale: float
    B2: Optional[torch.Tensor] = None  # second weight operand, B's shape
    a_scale_inv: Optional[torch.Tensor] = None  # FP8 dequantisation factors, 1 fp32 each
    b_scale_inv: Optional[torch.Tensor] = None
    col_scale: Optional[torch.Tensor] = None    # fp32, one per output column
    row_stat: Optional[torch.Tensor] = None     # fp32, one per row (the forward's S)
    row_scale: Optional[torch.Tensor] = None    # fp32, one per row (batch x M): the consumed S
    extra: dict = field(default_factory=dict)


def _bias_len(w: Workload) -> int:
    prog = list(w.program)
    if "bias" not in prog:
        return 0
    ib = prog.index("bias")
    ip = next((i for i, op in enumerate(prog) if op.startswith("pair_") or op.startswith("dswiglu")), None)
    return w.N if (ip is None or ib < ip) else w.n_out


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None) -> Inputs:
    """Draws the workload's tensors with a generator on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(1000 + w.index if seed is None else seed)

    def draw(shape, std, dtype=torch.bfloat16):
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        t.mul_(std)
        return t.to(dtype)

    def operand(shape, std, qscale, relu=False):
        if w.in_type == "bf16":
            t = draw(shape, std, torch.float32)
            return (t.clamp_min_(0) if relu else t).to(torch.bfloat16)
        t = draw(shape, std, torch.float32)
        if relu:
            t.clamp_min_(0)
        fmt = FP8_FORMATS[w.in_type]
        lim = torch.finfo(fmt).max
        return (t * qscale).clamp_(-lim, lim).to(fmt).view(torch.uint8)

    lead = (w.batch,) if w.batch > 1 else ()
    A = operand(lead + (w.M, w.K), w.a_std, w.a_qscale, w.a_relu)
    nbc = w.N // 2 if w.dual else w.N
    B = operand(lead + ((w.K, nbc) if w.b_layout == "kn" else (nbc, w.K)), w.b_std, w.b_qscale)
    nb = _bias_len(w)
    bias = draw((nb,), w.bias_std, torch.float32) if nb else None
    aux = draw(lead + (w.M, w.n_out), w.aux_std) if w.aux else None
    B2 = operand(tuple(B.shape), w.b_std, w.b_qscale) if w.dual else None
    inp = Inputs(A=A, B=B, bias=bias, aux=aux, alpha=w.alpha, fp8_scale=w.fp8_scale, B2=B2)
    if w.col_scale_std is not None:
        inp.col_scale = 1.0 + draw((w.n_out,), w.col_scale_std, torch.float32)
    if w.finish == "rmsnorm_backward":
        inp.row_stat = 1.0 + draw((w.M,), 0.05, torch.float32)
    if w.row_scale_std is not None:
        inp.row_scale = 1.0 + draw((w.batch * w.M,), w.row_scale_std, torch.float32)
    if w.in_type != "bf16":
        inp.a_scale_inv = torch.tensor([1.0 / w.a_qscale], dtype=torch.float32, device=device)
        inp.b_scale_inv = torch.tensor([1.0 / w.b_qscale], dtype=torch.float32, device=device)
    return inp


FP8_FORMATS = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
