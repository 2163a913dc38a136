"""Comparison rules between the CUDA path and the fp64 oracle.

Tolerances (as the benchmark statement fixes them, with the readings noted):
  bf16 outputs   |g - r| <= 2e-2 * max(|r|, 1e-2 * RMS(r))   (relative error
                 2e-2, floored at 1% of the tensor RMS so that zero crossings
                 of GELU / ReLU / gelu' do not divide by ~0)
  fp32 rows      relative 1e-3
  fp32 columns   |g - r| <= 1e-3 * sum_m |y[m, n]|
  AMAX           within one bf16 ulp of r
  e4m3 codes     identical, except two adjacent codes when the fp64 value lies
                 within one bf16 ulp (2^-8 relative) of the midpoint between them,
                 that ulp floored at 1% of the compared values' RMS like the
                 bf16 bound (a value from a cancellation near zero carries the
                 fp32 error of the tensor's scale, not of its own size)
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from gemm_epilogue_transformer_smem_gb300 import api, synth

BF16_TOL = 2e-2
RED_TOL = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


# Error reports of the comparisons made with report=..., printed at the end
# of the pytest run (tests/conftest.py): the floored bound decides pass or
# fail, the unfloored relative error is reported beside it.
REPORTS = []
NOTES = []  # one-line results printed beside them


def bf16_error_stats(g: np.ndarray, ref: np.ndarray) -> dict:
    """Unfloored relative error |g - r| / |r| over the elements with r != 0
    (its maximum, the count above 2e-2) and the largest ratio of the error to
    the floored bound that decides the test."""
    err = np.abs(g - ref)
    mag = np.abs(ref)
    nz = mag > 0
    rel = err[nz] / mag[nz]
    rms = math.sqrt(float(np.mean(ref * ref))) if ref.size else 0.0
    bound = BF16_TOL * np.maximum(mag, 1e-2 * rms)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    imax = int(np.argmax(rel)) if rel.size else -1
    return {"n": int(ref.size), "max_rel_unfloored": float(rel.max()) if rel.size else 0.0,
            "ref_at_max_rel": float(mag[nz][imax]) if rel.size else 0.0,
            "n_above_2e-2_unfloored": int(np.count_nonzero(rel > BF16_TOL)),
            "zeros_in_ref": int(ref.size - np.count_nonzero(nz)),
            "max_err_over_bound": float(ratio.max()) if ref.size else 0.0, "rms": rms}


def check_bf16(got_bits: np.ndarray, ref: np.ndarray, what="C", report=None):
    """Passes when |g - r| <= 2e-2 * max(|r|, 1e-2 * RMS(r)) everywhere.
    Returns the error statistics; with report="name" they are also kept for
    the end-of-run summary."""
    g = oracle.bf16_bits_to_f64(got_bits)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    if ref.size == 0:
        return None
    stats = bf16_error_stats(g, ref)
    if report:
        REPORTS.append((report, what, stats))
    rms = stats["rms"]
    bound = BF16_TOL * np.maximum(np.abs(ref), 1e-2 * rms)
    err = np.abs(g - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d elements outside tolerance; first %s: got %s want %s" % (
            what, int(bad.sum()), bad.size, idx.tolist(), g[tuple(idx.T)].tolist(),
            ref[tuple(idx.T)].tolist()))
    return stats


def check_e4m3(got: np.ndarray, want_codes: np.ndarray, ref_scaled: np.ndarray):
    """Returns the number of codes that differ (each one adjacent to the
    oracle's and at a rounding boundary within the tolerance)."""
    got = np.asarray(got, dtype=np.uint8)
    want = np.asarray(want_codes, dtype=np.uint8)
    assert got.shape == want.shape
    zero = lambda c: (c & 0x7F) == 0
    diff = (got != want) & ~(zero(got) & zero(want))
    if not diff.any():
        return 0
    ref_scaled = np.asarray(ref_scaled, dtype=np.float64)
    floor = 1e-2 * math.sqrt(float(np.mean(ref_scaled * ref_scaled)))
    for idx in np.argwhere(diff):
        i = tuple(idx)
        dg = float(oracle.e4m3_to_f64([got[i]])[0])
        dw = float(oracle.e4m3_to_f64([want[i]])[0])
        r = float(ref_scaled[i])
        lo, hi = min(dg, dw), max(dg, dw)
        # adjacent: no representable value strictly between them
        between = oracle.to_e4m3([(lo + hi) / 2])[0]
        mid = (lo + hi) / 2
        adjacent = oracle.e4m3_to_f64([between])[0] in (lo, hi)
        near = abs(r - mid) <= 2.0 ** -8 * max(abs(mid), floor, 2.0 ** -9)
        assert adjacent and near, "e4m3 code %s: got %#x want %#x for value %r" % (
            i, got[i], want[i], r)
    return int(diff.sum())


def bf16_ulp(x: float) -> float:
    if x == 0:
        return 2.0 ** -133
    return 2.0 ** (math.floor(math.log2(abs(x))) - 7)


def check_amax(got: float, ref: float):
    assert abs(got - ref) <= bf16_ulp(ref), (got, ref)


def check_rows(got: np.ndarray, ref: np.ndarray):
    np.testing.assert_allclose(np.asarray(got, np.float64), ref, rtol=RED_TOL, atol=0)


def check_cols(got: np.ndarray, ref: np.ndarray, abs_sum: np.ndarray):
    err = np.abs(np.asarray(got, np.float64) - ref)
    bad = err > RED_TOL * abs_sum
    assert not bad.any(), "column sums: %d bad, first %s" % (int(bad.sum()), np.argwhere(bad)[:5].tolist())


# ------------------------------------------------------------------ running

def operand_host(t: torch.Tensor, in_type: str) -> np.ndarray:
    """Host copy of an operand as the oracle reads it: bf16 bit patterns or
    FP8 codes."""
    if t is None:
        return None
    return bits(t) if in_type == "bf16" else t.detach().contiguous().cpu().numpy()


def scalar(t):
    return 1.0 if t is None else float(t.item())


def oracle_problem(w: synth.Workload, inp: synth.Inputs) -> oracle.Problem:
    prog = list(w.program)
    aux = bits(inp.aux) if inp.aux is not None else None
    return oracle.Problem(
        A=operand_host(inp.A, w.in_type), B=operand_host(inp.B, w.in_type), program=prog,
        b_is_nk=(w.b_layout == "nk"),
        alpha=inp.alpha, bias=None if inp.bias is None else inp.bias.detach().cpu().numpy(),
        residual=aux if w.aux == "residual" else None,
        preact=aux if w.aux == "preact" else None, fp8_scale=inp.fp8_scale,
        B2=operand_host(inp.B2, w.in_type), a_type=w.in_type, b_type=w.in_type,
        a_scale_inv=scalar(inp.a_scale_inv), b_scale_inv=scalar(inp.b_scale_inv),
        col_scale=None if inp.col_scale is None else inp.col_scale.detach().cpu().numpy(),
        row_scale=None if inp.row_scale is None else inp.row_scale.detach().cpu().numpy())


def run_cuda(w: synth.Workload, inp: synth.Inputs, unfused=False, **kw):
    plan = api.Plan(w.M, w.N, w.K, w.program, b_layout=w.b_layout, dual=w.dual, a_type=w.in_type,
                    b_type=w.in_type, batch=w.batch)
    out = api.allocate_outputs(plan, inp.A.device)
    scratch = None
    if unfused:
        scratch = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=inp.A.device)
    api.run_program(plan, inp.A, inp.B, out, alpha=inp.alpha, fp8_scale=inp.fp8_scale,
                    bias=inp.bias, aux=inp.aux, unfused_scratch=scratch, B2=inp.B2,
                    a_scale_inv=inp.a_scale_inv, b_scale_inv=inp.b_scale_inv, col_scale=inp.col_scale,
                    row_scale=inp.row_scale, **kw)
    torch.cuda.synchronize()
    status = plan.query_status(out.workspace)
    assert status == 0, "kernel status %d" % status
    return plan, out


def compare_rows(w, inp, out, rows=None, oracle_p=None, report=None):
    """Full output rows (all columns) of the listed rows, every output the
    program has; `rows` None = all rows."""
    p = oracle_p or oracle_problem(w, inp)
    ref = p.rows(rows)
    sel = slice(None) if rows is None else torch.as_tensor(np.asarray(rows), device=out.workspace.device)
    prog = [op.partition(":")[0] for op in w.program]
    if out.C is not None:
        check_bf16(bits(out.C[sel]), ref["y"], "C rows", report=report)
    if out.C8 is not None:
        check_e4m3(out.C8[sel].cpu().numpy(), ref["c_e4m3"], ref["y"] * inp.fp8_scale)
    if out.row_out is not None and "row_dot" in prog:
        # sum_n y x can cancel: bound by the sum of the magnitudes of its terms
        check_cols(out.row_out[sel].cpu().numpy(), ref["row_stat"], row_dot_abs(w, inp, ref, rows))
    elif out.row_out is not None:
        check_rows(out.row_out[sel].cpu().numpy(), ref["row_stat"])
    if "amax" in prog and rows is None:
        check_amax(float(out.amax.item()), ref["amax"])
    return ref


def row_dot_abs(w, inp, ref, rows):
    """sum_n |w[n] y[m,n] x[m,n]| for the row_dot of the drmsnorm program
    (store_bf16, col_scale, row_dot), from the oracle's stored values."""
    x = oracle.bf16_bits_to_f64(bits(inp.aux if rows is None else inp.aux[torch.as_tensor(np.asarray(rows))]))
    cs = inp.col_scale.detach().cpu().numpy().astype(np.float64)
    return np.abs(ref["y"] * cs[None, :] * x).sum(1)


def run_finish(w, inp, out):
    """The workload's second pass (gemm_epi_rmsnorm_backward) on the GEMM's
    outputs: returns (dx, dw) device tensors."""
    dx = torch.empty(out.C.shape, dtype=torch.bfloat16, device=out.C.device)
    dw = torch.empty(out.C.shape[1], dtype=torch.float32, device=out.C.device)
    api.rmsnorm_backward(out.C, inp.aux, inp.row_stat, out.row_out, w=inp.col_scale, dx=dx, dw=dw)
    torch.cuda.synchronize()
    return dx, dw


def compare_cols(w, inp, out, cols, oracle_p=None, report=None):
    p = oracle_p or oracle_problem(w, inp)
    ref = p.cols(cols)
    idx = torch.as_tensor(np.asarray(cols), device=out.workspace.device)
    if out.C is not None:
        check_bf16(bits(out.C[:, idx]), ref["y"], "C columns", report=report)
    if out.col_out is not None:
        check_cols(out.col_out[idx].cpu().numpy(), ref["col_stat"], np.abs(ref["y"]).sum(0))
    return ref
