"""Element offsets past 2^31 (needs a GB300 and about 13 GB of device memory).

The largest tensors here have 65600 x 32776 elements (4.3 GB of bf16), so
row offsets near the end exceed 2^31 elements and every address computed in
32-bit arithmetic would wrap.  N = 32770 is not a multiple of 8, so the last
two columns of every row go through the kernels' element-wise edge paths
(direct bf16 stores in the GEMM epilogue, partial copies in the RMSNorm
backward), again at offsets past 2^31.  Sampled rows are compared with the
oracle; padding columns must stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_epilogue_transformer_smem_gb300 import api

from parity import bits, check_bf16, check_cols, check_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"
M, N, LD = 65600, 32770, 32776
assert M * LD > 2 ** 31


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield cuda_lib
    torch.cuda.empty_cache()


def _sample_rows():
    rng = np.random.default_rng(31)
    tail = np.arange(M - 40, M)  # offsets past 2^31
    return np.unique(np.concatenate([[0, 1, 65535, 65536], rng.choice(M, 24, replace=False), tail]))


def test_gemm_epilogue_past_32_bit_offsets():
    """residual add + bf16 store + row RMS, K = 64."""
    K = 64
    g = torch.Generator(device=DEV).manual_seed(64)
    A = torch.randn(M, K, generator=g, device=DEV, dtype=torch.bfloat16)
    B = (torch.randn(K, LD, generator=g, device=DEV) / 8).to(torch.bfloat16)
    res = torch.randn(M, LD, generator=g, device=DEV, dtype=torch.bfloat16)
    C = torch.full((M, LD), 3.0, device=DEV, dtype=torch.bfloat16)
    prog = ["residual", "store_bf16", "row_rms:1e-6"]
    plan = api.Plan(M, N, K, prog, ldb=LD, ldc=LD, ld_aux=LD)
    row_out = torch.empty(M, device=DEV)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=DEV)
    plan.run(A, B, residual=res, C=C, row_out=row_out, workspace=ws)
    torch.cuda.synchronize()
    assert plan.query_status(ws) == 0
    assert torch.all(C[:, N:] == 3.0), "C written past N"
    rows = _sample_rows()
    idx = torch.as_tensor(rows, device=DEV)
    ref = oracle.Problem(bits(A[idx]), bits(B[:, :N]), prog, residual=bits(res[idx, :N])).rows()
    check_bf16(bits(C[idx, :N]), ref["y"], "C")
    check_rows(row_out[idx].cpu().numpy(), ref["row_stat"])
    del A, B, res, C


def test_backward_epilogue_past_32_bit_offsets():
    """gelu' of the pre-activation + bf16 store + column sums (the backward
    program's compiled kernel, column sums through TMEM), K = 64, W stored
    N x K: pre-activation loads and stores at offsets past 2^31, and column
    sums over all 65600 rows."""
    K = 64
    g = torch.Generator(device=DEV).manual_seed(66)
    A = torch.randn(M, K, generator=g, device=DEV, dtype=torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device=DEV) / 8).to(torch.bfloat16)
    pre = torch.randn(M, LD, generator=g, device=DEV, dtype=torch.bfloat16)
    C = torch.full((M, LD), 3.0, device=DEV, dtype=torch.bfloat16)
    prog = ["gelu_tanh_grad", "store_bf16", "col_sum"]
    plan = api.Plan(M, N, K, prog, b_layout="nk", ldc=LD, ld_aux=LD)
    col_out = torch.empty(N, device=DEV)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=DEV)
    plan.run(A, W, preact=pre, C=C, col_out=col_out, workspace=ws)
    torch.cuda.synchronize()
    assert plan.query_status(ws) == 0
    assert torch.all(C[:, N:] == 3.0), "C written past N"
    rows = _sample_rows()
    idx = torch.as_tensor(rows, device=DEV)
    p_rows = oracle.Problem(bits(A[idx]), bits(W), prog, b_is_nk=True, preact=bits(pre[idx, :N]))
    check_bf16(bits(C[idx, :N]), p_rows.rows()["y"], "C")
    # Columns are independent: the oracle takes just the sampled columns of W
    # and of the pre-activation, over every row.
    cols = torch.as_tensor([0, 31, 32, 16383, 32767, 32768, 32769], device=DEV)
    p_cols = oracle.Problem(bits(A), bits(W[cols]), prog, b_is_nk=True, preact=bits(pre[:, cols]))
    ref = p_cols.cols(list(range(len(cols))))
    check_cols(col_out[cols].cpu().numpy(), ref["col_stat"], np.abs(ref["y"]).sum(0))
    del A, W, pre, C


def test_rmsnorm_backward_past_32_bit_offsets():
    g = torch.Generator(device=DEV).manual_seed(65)
    dy = torch.randn(M, LD, generator=g, device=DEV, dtype=torch.bfloat16)
    x = torch.randn(M, LD, generator=g, device=DEV, dtype=torch.bfloat16)
    s = 0.5 + torch.rand(M, generator=g, device=DEV)
    r = torch.randn(M, generator=g, device=DEV) * N ** 0.5
    w = 1.0 + 0.1 * torch.randn(N, generator=g, device=DEV)
    dx = torch.full((M, LD), 5.0, device=DEV, dtype=torch.bfloat16)
    dw = torch.empty(N, device=DEV)
    api.rmsnorm_backward(dy[:, :N], x[:, :N], s, r, w=w, dx=dx[:, :N], dw=dw)
    torch.cuda.synchronize()
    assert torch.all(dx[:, N:] == 5.0), "dx written past N"
    rows = _sample_rows()
    idx = torch.as_tensor(rows, device=DEV)
    want_dx, _ = oracle.rmsnorm_backward(bits(dy[idx, :N]), bits(x[idx, :N]), s[idx].cpu().numpy(),
                                         r[idx].double().cpu().numpy(), w=w.cpu().numpy(), want_dw=False)
    check_bf16(bits(dx[idx, :N]), want_dx, "dx")
    # dw over every row, for a few columns (the last two are the ragged group)
    cols = torch.as_tensor([0, 7, 8, 16383, 32767, 32768, 32769], device=DEV)
    terms = dy[:, cols].double() * x[:, cols].double() * s.double()[:, None]
    check_cols(dw[cols].cpu().numpy(), terms.sum(0).cpu().numpy(), terms.abs().sum(0).cpu().numpy())
    del dy, x, dx
