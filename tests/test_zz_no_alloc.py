"""gemm_epi_run_no_alloc: the entry point for callers that cannot allocate
device memory (a host framework or plugin interface that passes only input
and output pointers and owns every other allocation, or a latency-critical
loop that avoids cudaMalloc's implicit device synchronisation).  It keeps its
status words and row counters in a static array inside the library instead
of a caller-supplied workspace.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from gemm_epilogue_transformer_smem_gb300 import api, native, synth

from parity import (BF16_TOL, RED_TOL, bits, check_amax, check_bf16, check_cols, check_rows,
                    oracle_problem)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _call_no_alloc(lib, plan, args):
    s = torch.cuda.current_stream().cuda_stream
    return lib.gemm_epi_run_no_alloc(plan.handle, ctypes.byref(args), ctypes.c_void_p(s))


def test_no_alloc_matches_workspace_path_on_two_calls(cuda_lib):
    """Residual add + bf16 store + row RMS over several row and column tiles:
    the row statistics go through the per-row-tile counters in the scratch,
    so a second call only matches if the first call's counters were cleared.
    Both calls are checked against the fp64 oracle and against gemm_epi_run."""
    lib = cuda_lib
    w = synth.WORKLOADS["downproj"].scaled(384, 1000, 328)
    inp = synth.make_inputs(w, DEV)
    plan = api.Plan(w.M, w.N, w.K, w.program, b_layout=w.b_layout)
    ref_rows = oracle_problem(w, inp).rows()

    ref = api.allocate_outputs(plan, DEV)
    api.run_program(plan, inp.A, inp.B, ref, aux=inp.aux)
    torch.cuda.synchronize()
    assert plan.query_status(ref.workspace) == native.GEMM_EPI_OK
    r = ref.C.double()
    rms = float(r.pow(2).mean().sqrt())

    for call in range(2):
        out = api.allocate_outputs(plan, DEV)
        out.C.fill_(0)
        out.row_out.fill_(-1.0)
        a = plan.args(inp.A, inp.B, residual=inp.aux, C=out.C, row_out=out.row_out, workspace=None)
        status = _call_no_alloc(lib, plan, a)
        assert status == native.GEMM_EPI_OK, lib.gemm_epi_last_error()
        torch.cuda.synchronize()
        check_bf16(bits(out.C), ref_rows["y"], "call %d: C" % call)
        check_rows(out.row_out.cpu().numpy(), ref_rows["row_stat"])
        g = out.C.double()
        bound = BF16_TOL * torch.maximum(r.abs(), torch.full_like(r, 1e-2 * rms))
        assert torch.all((g - r).abs() <= bound), "call %d: C differs from gemm_epi_run" % call
        np.testing.assert_allclose(out.row_out.cpu().numpy(), ref.row_out.cpu().numpy(), rtol=RED_TOL)


def test_no_alloc_amax_and_column_sums_on_two_calls(cuda_lib):
    """A second op family: gelu' with AMAX, a bf16 store and column sums
    (B stored N x K).  AMAX and the column sums are zeroed by every call, so
    the second call matches the oracle only if nothing carries over."""
    lib = cuda_lib
    prog = ["gelu_tanh_grad", "amax", "store_bf16", "col_sum"]
    w = synth.Workload("noalloc_bwd", 4, 300, 776, 192, "nk", tuple(prog), a_std=1.0, b_std=0.1,
                       aux="preact")
    inp = synth.make_inputs(w, DEV, seed=404)
    plan = api.Plan(w.M, w.N, w.K, prog, b_layout="nk")
    p = oracle_problem(w, inp)
    rows = p.rows()
    cols = p.cols(list(range(w.n_out)))
    for call in range(2):
        out = api.allocate_outputs(plan, DEV)
        out.C.fill_(0)
        a = plan.args(inp.A, inp.B, preact=inp.aux, C=out.C, amax=out.amax, col_out=out.col_out, workspace=None)
        status = _call_no_alloc(lib, plan, a)
        assert status == native.GEMM_EPI_OK, lib.gemm_epi_last_error()
        torch.cuda.synchronize()
        check_bf16(bits(out.C), rows["y"], "call %d: C" % call)
        check_amax(float(out.amax.item()), rows["amax"])
        check_cols(out.col_out.cpu().numpy(), cols["col_stat"], np.abs(cols["y"]).sum(0))


def test_no_alloc_rejects_plans_beyond_its_scratch(cuda_lib):
    """The scratch holds (65536 - 256) / 4 = 16320 row-block counters and a
    plan needs ceil(M / 256) * 2 * batch of them."""
    lib = cuda_lib
    counters = (native.GEMM_EPI_NO_ALLOC_SCRATCH_BYTES - 256) // 4
    rows_max = counters * 128
    plan = api.Plan(rows_max + 1, 256, 64, ["store_bf16"])
    assert plan.workspace_bytes > native.GEMM_EPI_NO_ALLOC_SCRATCH_BYTES
    a = plan.args(None, None)
    status = _call_no_alloc(lib, plan, a)
    assert status == native.GEMM_EPI_ERR_WORKSPACE
    assert b"scratch" in lib.gemm_epi_last_error()
    ok = api.Plan(rows_max, 256, 64, ["store_bf16"])
    assert ok.workspace_bytes <= native.GEMM_EPI_NO_ALLOC_SCRATCH_BYTES
    # A batch of 8 divides the limit by 8.
    per = counters // (2 * 8) * 256
    big = api.Plan(per + 256, 256, 64, ["store_bf16"], batch=8)
    assert big.workspace_bytes > native.GEMM_EPI_NO_ALLOC_SCRATCH_BYTES
    status = _call_no_alloc(lib, big, big.args(None, None))
    assert status == native.GEMM_EPI_ERR_WORKSPACE
    assert b"with batch 8 M is limited to %d rows" % per in lib.gemm_epi_last_error()
    assert api.Plan(per, 256, 64, ["store_bf16"], batch=8).workspace_bytes <= native.GEMM_EPI_NO_ALLOC_SCRATCH_BYTES
