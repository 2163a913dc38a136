"""Batched GEMM + epilogue (the cuDNN Graph API tutorial's batched matmul with
an epilogue) against the oracle, one oracle problem per batch (needs a GB300).

Batches of 3 with a ragged M; B either per batch or shared by every batch
(batch stride 0); per-batch row scales, residual / pre-activation, row and
column statistics; one AMAX over the whole batch.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_epilogue_transformer_smem_gb300 import api, native

from parity import bits, check_amax, check_bf16, check_cols, check_e4m3, check_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"
VARIANTS = {"1sm": native.GEMM_EPI_DEBUG_FORCE_1SM, "2sm": native.GEMM_EPI_DEBUG_FORCE_2SM,
            "interp": native.GEMM_EPI_DEBUG_FORCE_INTERPRETER}
PROGRAMS = {
    "bias_gelu": (("alpha", "bias", "gelu_tanh", "amax", "store_bf16"), "kn"),
    "fp8": (("alpha", "bias", "relu", "amax", "store_bf16", "store_e4m3"), "kn"),
    "residual_rms": (("residual", "store_bf16", "row_rms:1e-6"), "nk"),
    "grad_colsum": (("row_scale", "gelu_tanh_grad", "store_bf16", "col_sum"), "nk"),
    # the backward workload's compiled program: column sums through TMEM
    "grad_colsum_static": (("gelu_tanh_grad", "store_bf16", "col_sum"), "nk"),
    "dswiglu": (("alpha", "dswiglu", "store_bf16", "amax"), "nk"),
    "rms_bwd": (("store_bf16", "col_scale", "row_dot"), "kn"),
}


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    assert torch.cuda.is_available()
    return cuda_lib


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("shared_b", [False, True])
@pytest.mark.parametrize("name", sorted(PROGRAMS))
@pytest.mark.parametrize("N", [528, 512])  # 512: a K x N B comes through the 4-D map of 64-column blocks
def test_batched_matches_per_batch_oracle(name, shared_b, variant, N):
    program, layout = PROGRAMS[name]
    Bt, M, K = 3, 200, 136
    g = torch.Generator(device=DEV).manual_seed(41)

    def rnd(*shape, std=0.3):
        return (torch.randn(*shape, generator=g, device=DEV) * std).to(torch.bfloat16)

    A = rnd(Bt, M, K)
    bshape = (K, N) if layout == "kn" else (N, K)
    B = rnd(*bshape) if shared_b else rnd(Bt, *bshape)
    n_out = api.out_cols(list(program), N)
    bias = torch.randn(N, generator=g, device=DEV) * 0.1
    aux = rnd(Bt, M, n_out, std=1.0)
    row_scale = torch.rand(Bt, M, generator=g, device=DEV) + 0.5
    col_scale = torch.rand(n_out, generator=g, device=DEV) + 0.5
    plan = api.Plan(M, N, K, program, b_layout=layout, batch=Bt, batch_stride_b=0 if shared_b else None)
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, alpha=0.75, fp8_scale=64.0, bias=bias, row_scale=row_scale, aux=aux,
                    col_scale=col_scale, debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0

    amax = 0.0
    for b in range(Bt):
        names = [op.partition(":")[0] for op in program]
        p = oracle.Problem(bits(A[b]), bits(B if shared_b else B[b]), list(program), b_is_nk=(layout == "nk"),
                           alpha=0.75, bias=bias.cpu().numpy(), row_scale=row_scale[b].cpu().numpy(),
                           residual=bits(aux[b]) if any(n in api.RESIDUAL_OPS for n in names) else None,
                           preact=bits(aux[b]) if any(n in api.PREACT_OPS for n in names) else None, fp8_scale=64.0,
                           col_scale=col_scale.cpu().numpy())
        r = p.rows()
        check_bf16(bits(out.C[b]), r["y"], "C[%d]" % b)
        if out.C8 is not None:
            check_e4m3(out.C8[b].cpu().numpy(), r["c_e4m3"], r["y"] * 64.0)
        if out.row_out is not None and "row_dot" in names:
            terms = r["y"] * col_scale.double().cpu().numpy()[None, :] * oracle.bf16_bits_to_f64(bits(aux[b]))
            check_cols(out.row_out[b].cpu().numpy(), r["row_stat"], np.abs(terms).sum(1))
        elif out.row_out is not None:
            check_rows(out.row_out[b].cpu().numpy(), r["row_stat"])
        if out.col_out is not None:
            cs = p.cols(list(range(n_out)))
            check_cols(out.col_out[b].cpu().numpy(), cs["col_stat"], np.abs(cs["y"]).sum(0))
        amax = max(amax, r["amax"])
    if out.amax is not None:
        check_amax(float(out.amax.item()), amax)


def test_moe8_full_size_sampled():
    """The moe8 workload at full size (8 experts, 2048 x 28672 x 4096 each,
    own weights): sampled rows of every expert against its own oracle
    problem, the last rows of the last expert among them."""
    from gemm_epilogue_transformer_smem_gb300 import synth
    from parity import run_cuda
    w = synth.WORKLOADS["moe8"]
    inp = synth.make_inputs(w, DEV)
    plan, out = run_cuda(w, inp)
    rng = np.random.default_rng(w.index)
    for b in range(w.batch):
        rows = np.unique(np.concatenate([rng.choice(w.M, 12, replace=False), [0, w.M - 1]]))
        p = oracle.Problem(bits(inp.A[b]), bits(inp.B[b]), list(w.program))
        r = p.rows(rows)
        idx = torch.as_tensor(rows, device=DEV)
        check_bf16(bits(out.C[b][idx]), r["y"], "C[%d]" % b)
