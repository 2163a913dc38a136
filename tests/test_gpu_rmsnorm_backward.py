"""RMSNorm backward on the GPU: the GEMM epilogue's column scale and row
reduction, and the second pass (gemm_epi_rmsnorm_backward), against the
oracle through the C ABI (needs a GB300).

For y = x * S * w and upstream gradient dy (the GEMM's result):
  r[m] = sum_n w dy x                          (ROW_DOT in the GEMM epilogue)
  dx   = S w dy - x S^3 r / N (+ add)          (second pass)
  dw   = sum_m dy x S                          (second pass)
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_epilogue_transformer_smem_gb300 import api, synth

from parity import bits, check_bf16, check_cols, check_rows, compare_rows, oracle_problem, run_cuda, run_finish

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    assert torch.cuda.is_available()
    return cuda_lib


def _bf16(t):
    return t.to(torch.bfloat16)


# The last two shapes give each thread many rows (wide rows leave few row
# blocks; tall narrow ones many), so the per-thread copy ring wraps often.
@pytest.mark.parametrize("M,N,ld", [(300, 1003, 1008), (257, 4096, 4096), (1, 8, 8), (40, 2048 + 24, 2080),
                                    (1000, 32768 + 24, 32800), (20000, 259, 272)])
@pytest.mark.parametrize("with_w,with_add", [(True, True), (False, False)])
def test_second_pass_matches_oracle(M, N, ld, with_w, with_add):
    g = torch.Generator(device=DEV).manual_seed(100 + N)
    full = lambda std: _bf16(torch.randn(M, ld, generator=g, device=DEV) * std)  # noqa: E731
    dy, x, add = full(1.0), full(1.5), full(0.5)
    s = 0.5 + torch.rand(M, generator=g, device=DEV)
    r = torch.randn(M, generator=g, device=DEV) * N ** 0.5
    w = 1.0 + 0.1 * torch.randn(N, generator=g, device=DEV) if with_w else None
    dx = torch.full((M, ld), 7.0, dtype=torch.bfloat16, device=DEV)
    dw = torch.full((N,), 7.0, dtype=torch.float32, device=DEV)
    api.rmsnorm_backward(dy[:, :N], x[:, :N], s, r, w=w, add=add[:, :N] if with_add else None, dx=dx[:, :N], dw=dw)
    torch.cuda.synchronize()
    want_dx, want_dw = oracle.rmsnorm_backward(bits(dy[:, :N]), bits(x[:, :N]), s.cpu().numpy(),
                                               r.double().cpu().numpy(), w=None if w is None else w.cpu().numpy(),
                                               add=bits(add[:, :N]) if with_add else None)
    check_bf16(bits(dx[:, :N]), want_dx, "dx")
    assert torch.all(dx[:, N:] == 7.0), "dx written beyond N"
    xd = oracle.bf16_bits_to_f64(bits(x[:, :N]))
    dyd = oracle.bf16_bits_to_f64(bits(dy[:, :N]))
    check_cols(dw.cpu().numpy(), want_dw, np.abs(dyd * xd * s.double().cpu().numpy()[:, None]).sum(0))


def test_second_pass_optional_outputs():
    M, N = 64, 512
    g = torch.Generator(device=DEV).manual_seed(110)
    dy, x = _bf16(torch.randn(M, N, generator=g, device=DEV)), _bf16(torch.randn(M, N, generator=g, device=DEV))
    s = torch.ones(M, device=DEV)
    r = torch.randn(M, generator=g, device=DEV)
    dx = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    dw = torch.full((N,), 3.0, device=DEV)
    api.rmsnorm_backward(dy, x, s, r, dw=dw)            # dw only (overwritten, not accumulated)
    api.rmsnorm_backward(dy, x, s, r, dx=dx)            # dx only, w = 1
    torch.cuda.synchronize()
    want_dx, want_dw = oracle.rmsnorm_backward(bits(dy), bits(x), s.cpu().numpy(), r.double().cpu().numpy())
    check_bf16(bits(dx), want_dx, "dx")
    np.testing.assert_allclose(dw.cpu().numpy(), want_dw, rtol=1e-4, atol=1e-4)


def test_rejects_bad_arguments():
    M, N = 8, 24
    dy = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    s = torch.ones(M, device=DEV)
    with pytest.raises(Exception, match="MISALIGNED"):
        api.rmsnorm_backward(dy[:, 1:17], dy[:, :16], s, s, dx=dy[:, :16])   # base not 16-byte aligned
    with pytest.raises(Exception, match="INVALID"):
        api.rmsnorm_backward(dy, dy, s, None, dx=dy)                         # dx needs r


def check_dx_propagated(dx_bits, want_dx, gpu_dy_bits, oracle_dy_bits, gpu_r, oracle_r, x_bits, S, cs, N):
    """dx against the oracle's chain, with the stage-1 differences carried
    through: the stored dy may differ from the oracle's by one bf16 rounding
    (fp32 vs fp64 accumulator) and r by the reduction's fp32 error, and
    dx = S w dy - x S^3 r / N moves by S |w| |d dy| + |x| S^3 |d r| / N."""
    d_dy = np.abs(oracle.bf16_bits_to_f64(gpu_dy_bits) - oracle.bf16_bits_to_f64(oracle_dy_bits))
    d_r = np.abs(np.asarray(gpu_r, np.float64) - oracle_r)
    x = oracle.bf16_bits_to_f64(x_bits)
    prop = S[:, None] * np.abs(cs)[None, :] * d_dy + np.abs(x) * (S ** 3 * d_r / N)[:, None]
    g = oracle.bf16_bits_to_f64(dx_bits)
    rms = float(np.sqrt(np.mean(want_dx ** 2)))
    bound = 2e-2 * np.maximum(np.abs(want_dx), 1e-2 * rms) + prop
    bad = np.abs(g - want_dx) > bound
    assert not bad.any(), "dx: %d of %d outside the propagated bound" % (int(bad.sum()), bad.size)


def test_drmsnorm_chain():
    """GEMM (store dy, scale by w, reduce against x) then the second pass,
    against the oracle's own two stages: stage 2 reads the oracle's stage-1
    dy (bf16) and r, never the GPU's."""
    w = synth.WORKLOADS["drmsnorm"].scaled(384, 1024, 512)
    inp = synth.make_inputs(w, DEV)
    plan, out = run_cuda(w, inp)
    dx, dw = run_finish(w, inp, out)
    p = oracle_problem(w, inp)
    r1 = compare_rows(w, inp, out, oracle_p=p)
    S = inp.row_stat.cpu().numpy()
    cs = inp.col_scale.cpu().numpy()
    want_dx, want_dw = oracle.rmsnorm_backward(r1["c_bf16"], bits(inp.aux), S, r1["row_stat"], w=cs)
    check_dx_propagated(bits(dx), want_dx, bits(out.C), r1["c_bf16"], out.row_out.cpu().numpy(), r1["row_stat"],
                        bits(inp.aux), S, cs, w.N)
    x = oracle.bf16_bits_to_f64(bits(inp.aux))
    dyd = oracle.bf16_bits_to_f64(r1["c_bf16"])
    check_cols(dw.cpu().numpy(), want_dw, np.abs(dyd * x * S[:, None]).sum(0))


def test_drmsnorm_full_size_sampled():
    """The full workload: sampled rows of dx against the oracle (from the
    oracle's stage 1 on those rows), and dw against sum_m dy x S computed in
    fp64 from the GPU's own dy over every row (an invariant at any size)."""
    w = synth.WORKLOADS["drmsnorm"]
    inp = synth.make_inputs(w, DEV)
    plan, out = run_cuda(w, inp)
    dx, dw = run_finish(w, inp, out)
    rows = np.unique(np.concatenate([np.random.default_rng(8).choice(w.M, 48, replace=False), [0, w.M - 1]]))
    p = oracle_problem(w, inp)
    r1 = compare_rows(w, inp, out, rows=rows, oracle_p=p)
    idx = torch.as_tensor(rows, device=DEV)
    S = inp.row_stat[idx].cpu().numpy()
    cs = inp.col_scale.cpu().numpy()
    want_dx, _ = oracle.rmsnorm_backward(r1["c_bf16"], bits(inp.aux[idx]), S, r1["row_stat"], w=cs, want_dw=False)
    check_dx_propagated(bits(dx[idx]), want_dx, bits(out.C[idx]), r1["c_bf16"], out.row_out[idx].cpu().numpy(),
                        r1["row_stat"], bits(inp.aux[idx]), S, cs, w.N)
    dyx = out.C.double() * inp.aux.double() * inp.row_stat.double()[:, None]
    ref = dyx.sum(0)
    bound = 1e-3 * dyx.abs().sum(0) + 1e-6
    assert torch.all((dw.double() - ref).abs() <= bound)
