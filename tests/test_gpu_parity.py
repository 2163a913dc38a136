"""CUDA path vs the fp64 oracle, through the C ABI (needs a GB300).

Small shapes are compared element by element in full; they span several
128 x 256 tiles and leave ragged M, N and K tails.  The five benchmark
workloads run at their full sizes, in the launch configuration the bench
times, and are compared on sampled whole rows and whole columns plus
invariants that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_epilogue_transformer_smem_gb300 import api, native, synth

import parity
from parity import (bf16_ulp, bits, check_amax, check_bf16, check_cols, check_e4m3, check_rows, compare_cols,
                    compare_rows, oracle_problem, run_cuda)

pytestmark = pytest.mark.gpu

DEV = "cuda"
W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return cuda_lib


def small(name, M, N, K):
    return W[name].scaled(M, N, K)


# ------------------------------------------------------------ full compare, small

SMALL_SHAPES = [
    ("tiny", 64, 64, 128),          # the tiny workload itself (one partial tile)
    ("tiny", 300, 600, 200),        # 3 x 3 tiles, ragged M, N and K tails
    ("swiglu", 260, 1040, 136),     # pair op, 5 N tiles with a 16-column tail
    ("fp8", 257, 528, 264),         # FP8 store + AMAX, 16-column N tail, K tail of 8
    ("downproj", 384, 1000, 328),   # residual + row RMS across 4 N tiles
    ("backward", 200, 776, 192),    # B stored N x K, gelu' + column sums
    ("swiglu2w", 300, 768, 200),    # separate gate / up weights, 384 output columns
    ("fp8in", 257, 528, 272),       # e4m3 operands, K tail of 16 (one 16-byte group)
    ("dswiglu", 300, 520, 200),     # SwiGLU backward: 1040 output columns, 8-column N tail
    ("drmsnorm", 300, 1000, 200),   # dy stored, column scale, row dot with x
    # N a multiple of 64: B (K x N) comes through the 4-D map, one load per K block
    ("swiglu", 260, 1024, 136),     # 4 N tiles, K tail of 8
    ("fp8", 257, 576, 264),         # a last N tile of 64 columns (the rest of its blocks out of range)
]


# The two main-loop shapes: one CTA per 128 x 256 tile, or a CTA pair per
# 256 x 256 tile (the default whenever M > 128); and the op-interpreting
# kernel in place of a program's compiled one.
VARIANTS = {"1sm": native.GEMM_EPI_DEBUG_FORCE_1SM, "2sm": native.GEMM_EPI_DEBUG_FORCE_2SM,
            "interp": native.GEMM_EPI_DEBUG_FORCE_INTERPRETER,
            "interp1sm": native.GEMM_EPI_DEBUG_FORCE_INTERPRETER | native.GEMM_EPI_DEBUG_FORCE_1SM}


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("name,M,N,K", SMALL_SHAPES)
def test_small_full_compare(name, M, N, K, variant):
    w = small(name, M, N, K) if (M, N, K) != (W[name].M, W[name].N, W[name].K) else W[name]
    inp = synth.make_inputs(w, DEV)
    plan, out = run_cuda(w, inp, debug_flags=VARIANTS[variant])
    compare_rows(w, inp, out)
    if out.col_out is not None:
        compare_cols(w, inp, out, list(range(w.n_out)))


def unfused_oracle(w, inp):
    """The unfused baseline's own definition: the bare GEMM rounded to bf16,
    then the epilogue program applied to that stored tensor (written as the
    oracle's GEMM of the stored tensor with an exact bf16 identity)."""
    p = oracle_problem(w, inp)
    stored = oracle.Problem(p.A, p.B, ["store_bf16"], b_is_nk=p.b_is_nk, a_type=p.a_type, b_type=p.b_type,
                            a_scale_inv=p.a_scale_inv, b_scale_inv=p.b_scale_inv).rows()["c_bf16"]
    eye = oracle.to_bf16_bits(np.eye(w.N))
    p.A, p.B, p.b_is_nk = stored, eye, False
    p.a_type = p.b_type = "bf16"
    p.a_scale_inv = p.b_scale_inv = 1.0
    return p


@pytest.mark.parametrize("form", ["static", "interp"])
@pytest.mark.parametrize("name,M,N,K", [s for s in SMALL_SHAPES[1:] if s[0] != "swiglu2w"])
def test_small_unfused_baseline(name, M, N, K, form):
    """The separate pass, compiled for the program and interpreted."""
    w = small(name, M, N, K)
    inp = synth.make_inputs(w, DEV)
    flags = native.GEMM_EPI_DEBUG_FORCE_INTERPRETER if form == "interp" else 0
    plan, out = run_cuda(w, inp, unfused=True, debug_flags=flags)
    p = unfused_oracle(w, inp)
    compare_rows(w, inp, out, oracle_p=p)
    if out.col_out is not None:
        compare_cols(w, inp, out, list(range(w.n_out)), oracle_p=p)


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("program,layout", [
    (("store_bf16",), "kn"),
    (("store_bf16",), "nk"),
    (("alpha", "bias", "silu", "store_bf16"), "nk"),
    (("row_scale", "gelu_tanh", "amax", "store_bf16"), "kn"),
    (("alpha", "bias", "pair_swiglu", "store_bf16", "amax"), "kn"),
    (("pair_swiglu:4", "store_bf16"), "kn"),
    (("pair_swiglu:32", "relu", "store_bf16", "col_sum"), "nk"),
    (("residual", "gelu_tanh", "store_bf16", "store_e4m3", "row_rms_unrounded:1e-5"), "nk"),
    (("gelu_tanh_grad", "amax", "store_bf16", "col_sum", "row_rms"), "kn"),
    (("row_scale", "pair_mul", "store_bf16"), "kn"),
    (("row_scale", "pair_swiglu", "store_bf16"), "kn"),
    (("pair_mul:8", "amax", "store_bf16"), "nk"),
])
def test_program_variants(program, layout, variant):
    aux = "residual" if "residual" in program else ("preact" if "gelu_tanh_grad" in program else None)
    w = synth.Workload("variant", 11, 200, 512 + 64, 136, layout, program, a_std=0.3, b_std=0.3,
                       bias_std=0.1 if "bias" in program else None, aux=aux, alpha=0.75, fp8_scale=64.0)
    inp = synth.make_inputs(w, DEV, seed=77)
    row_scale = torch.rand(w.M, device=DEV) + 0.5
    plan = api.Plan(w.M, w.N, w.K, program, b_layout=layout)
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, inp.A, inp.B, out, alpha=inp.alpha, fp8_scale=inp.fp8_scale, bias=inp.bias,
                    row_scale=row_scale, aux=inp.aux, debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    p = oracle_problem(w, inp)
    p.row_scale = row_scale.cpu().numpy()
    compare_rows(w, inp, out, oracle_p=p)
    if out.col_out is not None:
        compare_cols(w, inp, out, list(range(w.n_out)), oracle_p=p)


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("program", [("pair_swiglu:128", "store_bf16"),
                                     ("row_scale", "pair_mul:128", "store_bf16"),
                                     ("alpha", "pair_swiglu:128", "amax", "store_bf16", "col_sum")])
def test_two_weight_programs(program, layout, variant):
    """Separate gate / up weights (GEMM_EPI_B_DUAL): out = f(X@B) * (X@B2)."""
    w = synth.Workload("two_weight", 13, 260, 1280, 136, layout, program, a_std=0.3, b_std=0.3,
                       alpha=0.75, dual=True)
    inp = synth.make_inputs(w, DEV, seed=31)
    row_scale = torch.rand(w.M, device=DEV) + 0.5
    plan = api.Plan(w.M, w.N, w.K, program, b_layout=layout, dual=True)
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, inp.A, inp.B, out, alpha=inp.alpha, row_scale=row_scale, B2=inp.B2,
                    debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    p = oracle_problem(w, inp)
    p.row_scale = row_scale.cpu().numpy()
    compare_rows(w, inp, out, oracle_p=p)
    if out.col_out is not None:
        compare_cols(w, inp, out, list(range(w.n_out)), oracle_p=p)


@pytest.mark.parametrize("pair", ["pair_mul", "pair_swiglu"])
def test_rmsnorm_mlp_chain(pair):
    """The RMSNorm-MLP chain of the Superoptimizer page (section 10) without a
    separate scale kernel: a down-projection emits out = residual + X@W1 and
    S = 1/sqrt(mean(out^2) + eps) from its epilogue; the next GEMM consumes
    out with S as a row scale, (out*S)@W2 = (out@W2)*S, and pairs gate/up
    (plain product, or SwiGLU).  Each stage's oracle reads the oracle's own
    stage-1 results, never the GPU's."""
    g = torch.Generator(device=DEV).manual_seed(21)
    M, K1, H, N2 = 384, 512, 1024, 1536
    X = (torch.randn(M, K1, generator=g, device=DEV) / K1 ** 0.5).to(torch.bfloat16)
    W1 = (torch.randn(K1, H, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
    R = torch.randn(M, H, generator=g, device=DEV).to(torch.bfloat16)
    W2 = (torch.randn(H, N2, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
    prog1 = ["residual", "store_bf16", "row_rms:1e-6"]
    prog2 = ["row_scale", pair, "store_bf16"]
    p1 = api.Plan(M, H, K1, prog1)
    o1 = api.allocate_outputs(p1, DEV)
    api.run_program(p1, X, W1, o1, aux=R)
    p2 = api.Plan(M, N2, H, prog2)
    o2 = api.allocate_outputs(p2, DEV)
    api.run_program(p2, o1.C, W2, o2, row_scale=o1.row_out)
    torch.cuda.synchronize()
    assert p1.query_status(o1.workspace) == 0 and p2.query_status(o2.workspace) == 0
    r1 = oracle.Problem(bits(X), bits(W1), prog1, residual=bits(R)).rows()
    check_rows(o1.row_out.cpu().numpy(), r1["row_stat"])
    S = r1["row_stat"].astype(np.float32)
    r2 = oracle.Problem(r1["c_bf16"], bits(W2), prog2, row_scale=S).rows()
    # Stage 1 rounds out to bf16 from fp32 on the GPU and from fp64 in the
    # oracle, so a few stage-2 inputs differ by one bf16 ulp.  Carried through
    # the GEMM (|W2|), the row scale and the pair op (|silu'| <= 1.1), that
    # bounds the extra stage-2 difference per element; it is added to the
    # bf16 tolerance of a single stage.
    Xr = oracle.bf16_bits_to_f64(r1["c_bf16"])
    with np.errstate(divide="ignore"):
        ulp = np.where(Xr != 0, 2.0 ** (np.floor(np.log2(np.abs(Xr))) - 7), 0.0)
    E = (ulp @ np.abs(oracle.bf16_bits_to_f64(bits(W2)))) * S[:, None]  # M x N2 accumulator bound
    acc = oracle.Problem(r1["c_bf16"], bits(W2), ["row_scale"], row_scale=S).rows()["y"]
    ag, au, Eg, Eu = acc[:, 0::2], acc[:, 1::2], E[:, 0::2], E[:, 1::2]
    if pair == "pair_mul":
        fg, dfg = np.abs(ag), 1.0
    else:
        fg, dfg = np.abs(ag / (1 + np.exp(-ag))), 1.1
    prop = dfg * Eg * np.abs(au) + fg * Eu + dfg * Eg * Eu
    g2 = oracle.bf16_bits_to_f64(bits(o2.C))
    rms = float(np.sqrt(np.mean(r2["y"] ** 2)))
    bound = 2e-2 * np.maximum(np.abs(r2["y"]), 1e-2 * rms) + prop
    bad = np.abs(g2 - r2["y"]) > bound
    assert not bad.any(), "chain output: %d of %d outside the propagated bound" % (int(bad.sum()), bad.size)


# ------------------------------------------------------------ exact pins on the GPU

def test_integer_inputs_bit_exact():
    """Small integers keep the fp32 accumulation exact, and |C| <= 256 keeps
    the bf16 store exact: any difference is a bug."""
    g = torch.Generator(device=DEV).manual_seed(5)
    M, N, K = 256, 512, 320
    A = torch.randint(-2, 3, (M, K), generator=g, device=DEV).to(torch.bfloat16)
    B = torch.randint(-2, 3, (K, N), generator=g, device=DEV).to(torch.bfloat16)
    plan = api.Plan(M, N, K, ["store_bf16"])
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out)
    torch.cuda.synchronize()
    ref = oracle.Problem(bits(A), bits(B), ["store_bf16"]).rows()
    assert np.abs(ref["y"]).max() <= 256
    assert np.array_equal(bits(out.C), ref["c_bf16"])


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_identity_and_permutation(layout):
    K, N = 256, 384
    g = torch.Generator(device=DEV).manual_seed(6)
    B = torch.randn((K, N) if layout == "kn" else (N, K), generator=g, device=DEV).to(torch.bfloat16)
    Bkn = B if layout == "kn" else B.t().contiguous()
    perm = torch.randperm(K, generator=g, device=DEV)
    for A in (torch.eye(K, device=DEV, dtype=torch.bfloat16),
              torch.eye(K, device=DEV, dtype=torch.bfloat16)[perm]):
        plan = api.Plan(K, N, K, ["store_bf16"], b_layout=layout)
        out = api.allocate_outputs(plan, DEV)
        api.run_program(plan, A, B, out)
        torch.cuda.synchronize()
        want = (A.float() @ Bkn.float()).to(torch.bfloat16)  # exact: one nonzero per row
        assert torch.equal(out.C.view(torch.int16), want.view(torch.int16))


def test_row_scale_rewrite_identity():
    """(X*S)@W == (X@W)*S for a row-broadcast S (powers of two: exact)."""
    g = torch.Generator(device=DEV).manual_seed(8)
    M, N, K = 300, 512, 192
    X = torch.randn(M, K, generator=g, device=DEV).to(torch.bfloat16)
    Wt = torch.randn(K, N, generator=g, device=DEV).to(torch.bfloat16)
    S = torch.pow(2.0, torch.randint(-3, 4, (M,), generator=g, device=DEV).float())
    p1 = api.Plan(M, N, K, ["store_bf16"])
    o1 = api.allocate_outputs(p1, DEV)
    api.run_program(p1, (X.float() * S[:, None]).to(torch.bfloat16), Wt, o1)
    p2 = api.Plan(M, N, K, ["row_scale", "store_bf16"])
    o2 = api.allocate_outputs(p2, DEV)
    api.run_program(p2, X, Wt, o2, row_scale=S)
    torch.cuda.synchronize()
    assert torch.equal(o1.C.view(torch.int16), o2.C.view(torch.int16))


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (1, 256, 8), (127, 264, 64), (129, 8, 72), (64, 64, 0),
                                   (300, 520, 0), (260, 296, 40), (129, 264, 520)])
def test_edge_shapes(M, N, K, variant):
    w = synth.Workload("edge", 12, M, N, K, "kn", ("alpha", "bias", "gelu_tanh", "amax", "store_bf16"),
                       a_std=0.5, b_std=0.5, bias_std=0.1, alpha=1.5)
    inp = synth.make_inputs(w, DEV, seed=99)
    plan, out = run_cuda(w, inp, debug_flags=VARIANTS[variant])
    compare_rows(w, inp, out)


def test_empty_problem_clears_reductions():
    plan = api.Plan(0, 64, 64, ["amax", "store_bf16", "col_sum"])
    out = api.allocate_outputs(plan, DEV)
    out.amax.fill_(7.0)
    out.col_out.fill_(7.0)
    A = torch.empty((0, 64), device=DEV, dtype=torch.bfloat16)
    B = torch.zeros((64, 64), device=DEV, dtype=torch.bfloat16)
    plan.run(A, B, C=out.C, amax=out.amax, col_out=out.col_out, workspace=out.workspace)
    torch.cuda.synchronize()
    assert out.amax.item() == 0.0 and torch.all(out.col_out == 0)


@pytest.mark.parametrize("variant", ["2sm", "interp"])
def test_fp8_codes_saturate_like_the_oracle(variant):
    """Outputs far beyond the e4m3 range: every code saturates to +-448
    (0x7E / 0xFE) exactly where the oracle's does, never to NaN."""
    M, N, K = 200, 272, 64  # e4m3 rows must start on 16-byte boundaries
    w = synth.Workload("sat", 13, M, N, K, "kn", ("alpha", "bias", "gelu_tanh", "amax", "store_bf16", "store_e4m3"),
                       a_std=1.0, b_std=1.0, bias_std=1.0, alpha=1.0, fp8_scale=1e4)
    inp = synth.make_inputs(w, DEV, seed=5)
    plan, out = run_cuda(w, inp, debug_flags=VARIANTS[variant])
    ref = compare_rows(w, inp, out)
    codes = out.C8.cpu().numpy()
    assert np.all(codes[ref["c_e4m3"] == 0x7E] == 0x7E) and np.all(codes[ref["c_e4m3"] == 0xFE] == 0xFE)
    assert (ref["c_e4m3"] == 0x7E).sum() > M * N // 4  # most codes saturated
    assert not np.any((codes & 0x7F) == 0x7F)  # no NaN codes


@pytest.mark.parametrize("variant", ["2sm", "interp"])
def test_nan_input_row_propagates_and_wins_amax(variant):
    """A NaN in one row of A makes that row's outputs NaN (bf16 NaN, e4m3 NaN
    code) and AMAX NaN: the integer maximum over float bits orders NaN above
    every finite value and infinity.  Every other row still matches the
    oracle."""
    M, N, K = 200, 272, 64
    prog = ["gelu_tanh", "amax", "store_bf16", "store_e4m3"]
    w = synth.Workload("nanrow", 14, M, N, K, "kn", tuple(prog), a_std=0.5, b_std=0.5, fp8_scale=8.0)
    inp = synth.make_inputs(w, DEV, seed=6)
    bad = 37
    inp.A[bad, 3] = float("nan")
    plan, out = run_cuda(w, inp, debug_flags=VARIANTS[variant])
    c = out.C.float()
    assert torch.isnan(c[bad]).all()
    assert np.all((out.C8[bad].cpu().numpy() & 0x7F) == 0x7F)
    assert np.isnan(out.amax.item())
    keep = [r for r in range(M) if r != bad]
    ref = oracle_problem(w, inp).rows(keep)
    check_bf16(bits(out.C[keep]), ref["y"])
    check_e4m3(out.C8[keep].cpu().numpy(), ref["c_e4m3"], ref["y"] * w.fp8_scale)


def test_zero_columns_launch_nothing_and_clear_amax():
    """N == 0: no output column, no launch; AMAX is still overwritten (0)."""
    M, K = 64, 64
    plan = api.Plan(M, 0, K, ["amax", "store_bf16", "col_sum"], ldb=8, ldc=8)
    amax = torch.full((1,), 7.0, device=DEV)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=DEV)
    A = torch.zeros((M, K), device=DEV, dtype=torch.bfloat16)
    B = torch.zeros((K, 8), device=DEV, dtype=torch.bfloat16)
    C = torch.full((M, 8), 3.0, device=DEV, dtype=torch.bfloat16)
    col = torch.full((8,), 5.0, device=DEV)
    plan.run(A, B, C=C, amax=amax, col_out=col, workspace=ws)
    torch.cuda.synchronize()
    assert plan.query_status(ws) == 0
    assert amax.item() == 0.0
    assert torch.all(C == 3.0)  # nothing written outside the (empty) output


@pytest.mark.parametrize("N", [300, 333, 7])
def test_strided_operands_and_guard_bands(N):
    """Row strides larger than the logical width and output widths that end
    inside a 16-byte group; sentinels beyond every declared extent survive."""
    M, K = 200, 136
    lda, ldb = K + 24, (N + 7) // 8 * 8 + 16
    ldc, ldc8 = (N + 7) // 8 * 8 + 32, (N + 15) // 16 * 16 + 32
    g = torch.Generator(device=DEV).manual_seed(3)
    Abuf = torch.randn(M, lda, generator=g, device=DEV).to(torch.bfloat16)
    Bbuf = torch.randn(K, ldb, generator=g, device=DEV).to(torch.bfloat16)
    Cbuf = torch.full((M + 3, ldc), 12345.0, device=DEV).to(torch.bfloat16)
    C8buf = torch.full((M + 3, ldc8), 0x5A, dtype=torch.uint8, device=DEV)
    sentinel = Cbuf[0, 0].clone()
    prog = ["gelu_tanh", "store_bf16", "store_e4m3"]
    plan = api.Plan(M, N, K, prog, lda=lda, ldb=ldb, ldc=ldc, ldc8=ldc8)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=DEV)
    plan.run(Abuf, Bbuf, C=Cbuf, C8=C8buf, fp8_scale=8.0, workspace=ws)
    torch.cuda.synchronize()
    assert plan.query_status(ws) == 0
    assert torch.all(Cbuf[:M, N:] == sentinel) and torch.all(Cbuf[M:] == sentinel)
    assert torch.all(C8buf[:M, N:] == 0x5A) and torch.all(C8buf[M:] == 0x5A)
    ref = oracle.Problem(bits(Abuf[:, :K]), bits(Bbuf[:, :N]), prog, fp8_scale=8.0).rows()
    check_bf16(bits(Cbuf[:M, :N]), ref["y"])
    from parity import check_e4m3
    check_e4m3(C8buf[:M, :N].cpu().numpy(), ref["c_e4m3"], ref["y"] * 8.0)


def test_misaligned_and_missing_buffers_rejected():
    plan = api.Plan(128, 256, 64, ["store_bf16", "amax"])
    out = api.allocate_outputs(plan, DEV)
    A = torch.zeros(128 * 64 + 8, device=DEV, dtype=torch.bfloat16)
    B = torch.zeros(64, 256, device=DEV, dtype=torch.bfloat16)
    with pytest.raises(native.GemmEpiError) as e:
        plan.run(A[1:], B, C=out.C, amax=out.amax, workspace=out.workspace)
    assert e.value.status == native.GEMM_EPI_ERR_MISALIGNED
    with pytest.raises(native.GemmEpiError) as e:
        plan.run(A, B, C=out.C, amax=None, workspace=out.workspace)
    assert e.value.status == native.GEMM_EPI_ERR_INVALID_VALUE
    with pytest.raises(native.GemmEpiError) as e:
        plan.run(A, B, C=out.C, amax=out.amax, workspace=out.workspace[:16])
    assert e.value.status == native.GEMM_EPI_ERR_WORKSPACE


@pytest.mark.parametrize("hook", ["stage", "second_kblock"])
@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_bounded_wait_reports_timeout_and_context_survives(variant, hook):
    """Loads the producer deliberately never issues make the MMA warp's
    bounded wait run out; the kernel reports it and exits cleanly."""
    w = small("tiny", 512, 512, 256)
    inp = synth.make_inputs(w, DEV)
    plan = api.Plan(w.M, w.N, w.K, w.program)
    out = api.allocate_outputs(plan, DEV)
    flag = native.GEMM_EPI_DEBUG_SKIP_FIRST_LOAD if hook == "stage" else native.GEMM_EPI_DEBUG_SKIP_SECOND_LOAD
    api.run_program(plan, inp.A, inp.B, out, bias=inp.bias, timeout_ms=50, debug_flags=flag | VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == native.GEMM_EPI_ERR_TIMEOUT
    # Status words: [0] bit 0 a wait ran out, bit 1 the drain of the operand
    # loads after it also ran out; [1] the wait that ran out first (2: the
    # MMA warp's for the stage, 4: the epilogue's for the accumulator, which
    # started as early); [3] the stages the drain settled.
    #   stage: the first CTA never armed stage 0.  On the CTA-pair kernel the
    #     odd CTA still loaded into it: the drain arms it and waits for those
    #     bytes (bit 8); alone, nothing was loaded and nothing is settled.
    #   second_kblock: on the CTA pair, stage 0 (two K-blocks) is armed and
    #     one K-block short: the drain counts the missing bytes as arrived
    #     (bit 0); alone, that K-block is stage 1, never armed.
    words = out.workspace[:16].view(torch.int32).cpu().tolist()
    assert words[0] & 1 and not words[0] & 2, words
    assert words[1] in (2, 4), words
    if "1sm" in variant:
        assert words[3] == 0, words
    else:
        assert words[3] == (1 << 8 if hook == "stage" else 1), words
    # The context still works: a normal run afterwards is correct.
    api.run_program(plan, inp.A, inp.B, out, bias=inp.bias)
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    compare_rows(w, inp, out)


def test_graph_capture_replay_matches_eager():
    w = small("fp8", 512, 768, 256)
    inp = synth.make_inputs(w, DEV)
    plan = api.Plan(w.M, w.N, w.K, w.program)
    eager = api.allocate_outputs(plan, DEV)
    api.run_program(plan, inp.A, inp.B, eager, alpha=inp.alpha, fp8_scale=inp.fp8_scale, bias=inp.bias)
    torch.cuda.synchronize()
    out = api.allocate_outputs(plan, DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            api.run_program(plan, inp.A, inp.B, out, alpha=inp.alpha, fp8_scale=inp.fp8_scale,
                            bias=inp.bias)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.C.view(torch.int16), eager.C.view(torch.int16))
    assert torch.equal(out.C8, eager.C8)
    assert out.amax.item() == eager.amax.item()


# ------------------------------------------------------------ full-size workloads

FULL = ["tiny", "swiglu", "fp8", "downproj", "backward", "swiglu2w", "fp8in", "dswiglu", "drmsnorm",
        "rmsswiglu", "rmsglu", "decode"]


# Sampled rows and columns per workload: 512 of each for the SwiGLU,
# down-projection and backward configurations (the FP8 one is compared over
# every element below), fewer for the others.
SAMPLES = {"swiglu": (512, 512), "downproj": (512, 512), "backward": (512, 512)}


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_parity(name):
    w = W[name]
    inp = synth.make_inputs(w, DEV)
    plan, out = run_cuda(w, inp)
    rng = np.random.default_rng(w.index)
    want_rows, want_cols = SAMPLES.get(name, (96, 24))
    nrows = min(want_rows, w.M) if w.M > 128 else w.M
    rows = np.unique(np.concatenate([rng.choice(w.M, nrows, replace=False), [0, w.M - 1]]))
    p = oracle_problem(w, inp)
    ref = compare_rows(w, inp, out, rows=rows, oracle_p=p, report=name)
    ncols = min(want_cols, w.n_out) if w.n_out > 64 else w.n_out
    cols = np.unique(np.concatenate([rng.choice(w.n_out, ncols, replace=False), [0, w.n_out - 1]]))
    compare_cols(w, inp, out, cols, oracle_p=p, report=name)
    prog = [op.partition(":")[0] for op in w.program]
    # Invariants over the whole output.
    if "amax" in prog:
        amax = float(out.amax.item())
        cmax = out.C.float().abs().max().item()
        assert oracle.to_bf16_bits([amax])[0] == oracle.to_bf16_bits([cmax])[0]
        assert amax >= ref["amax"] * (1 - 2 ** -20)
    if "row_rms" in prog:
        c = out.C.float()
        r = torch.rsqrt(c.pow(2).mean(1, dtype=torch.float64) + 1e-6).float()
        torch.testing.assert_close(out.row_out, r, rtol=1e-5, atol=0)
    if "col_sum" in prog:
        c = out.C.double()
        s = c.sum(0)
        bound = 2.0 ** -8 * c.abs().sum(0) + 1e-6
        assert torch.all((out.col_out.double() - s).abs() <= bound)


def test_full_size_fp8_against_the_whole_oracle():
    """The FP8-training workload (M = N = K = 8192: ReLU(0.5 A@B + bias),
    AMAX, bf16 and e4m3 stores) against the fp64 oracle over every element,
    in row blocks.  AMAX feeds the next FP8 quantisation (the cuDNN Graph API
    tutorial's matmul epilogue), so the whole-tensor maximum is checked to one
    bf16 ulp of the fp64 value, not only through invariants and samples."""
    w = W["fp8"]
    inp = synth.make_inputs(w, DEV)
    plan, out = run_cuda(w, inp)
    p = oracle_problem(w, inp)
    amax = 0.0
    c8_mismatch = 0
    step = 1024
    for r0 in range(0, w.M, step):
        rows = list(range(r0, min(w.M, r0 + step)))
        ref = p.rows(rows)
        amax = max(amax, ref["amax"])
        check_bf16(bits(out.C[r0:r0 + len(rows)]), ref["y"], "C rows %d.." % r0,
                   report="fp8-full" if r0 == 0 else None)
        c8_mismatch += check_e4m3(out.C8[r0:r0 + len(rows)].cpu().numpy(), ref["c_e4m3"], ref["y"] * inp.fp8_scale)
        del ref
    parity.NOTES.append("fp8 whole tensor vs oracle: amax %r (oracle %r, one bf16 ulp %.3g); e4m3 codes "
                        "differing at a rounding boundary: %d of %d" % (
                            float(out.amax.item()), amax, bf16_ulp(amax), c8_mismatch, w.M * w.n_out))
    check_amax(float(out.amax.item()), amax)


# The store path's chunk that straddles the output edge (columns 512..543)
# and the chunks past it, in the static FP8 kernels (bf16 + e4m3 stores) and
# the bf16-only backward kernel.  A race between a chunk's TMA store and a
# later chunk's staging writes once left the straddling columns unwritten;
# repeated runs guard against its return.
@pytest.mark.parametrize("variant", ["1sm", "2sm"])
@pytest.mark.parametrize("name,N", [("fp8", 528), ("fp8", 536), ("backward", 520)])
def test_edge_chunk_stores_repeated(name, N, variant):
    w = small(name, 257 if name == "fp8" else 200, N, 264 if name == "fp8" else 192)
    inp = synth.make_inputs(w, DEV)
    cols = list(range(480, w.n_out))
    p = oracle_problem(w, inp)
    ref = p.cols(cols)
    ref8 = p.rows()["c_e4m3"][:, cols] if "store_e4m3" in w.program else None
    # e4m3 rows must start on 16-byte boundaries: a ragged e4m3 width gets a padded row stride
    ldc8 = (w.n_out + 15) // 16 * 16
    plan = api.Plan(w.M, w.N, w.K, w.program, b_layout=w.b_layout, ldc8=ldc8)
    out = api.allocate_outputs(plan, DEV)
    if out.C8 is not None:
        out.C8 = torch.empty((w.M, ldc8), dtype=torch.uint8, device=DEV)
    idx = torch.as_tensor(cols, device=DEV)
    for it in range(50):
        out.C.fill_(float("nan"))
        if out.C8 is not None:
            out.C8.fill_(0x7F)  # e4m3 NaN
        api.run_program(plan, inp.A, inp.B, out, alpha=inp.alpha, fp8_scale=inp.fp8_scale, bias=inp.bias,
                        aux=inp.aux, debug_flags=VARIANTS[variant])
        torch.cuda.synchronize()
        assert plan.query_status(out.workspace) == 0
        check_bf16(bits(out.C[:, idx]), ref["y"], "run %d, C columns 480.." % it)
        if ref8 is not None:
            check_e4m3(out.C8[:, idx].cpu().numpy(), ref8, ref["y"] * inp.fp8_scale)


@pytest.mark.parametrize("variant", ["1sm", "2sm", "interp"])
@pytest.mark.parametrize("name,M,N,K", [("swiglu", 520, 1040, 264), ("fp8", 520, 1040, 264),
                                        ("backward", 520, 1040, 264), ("dswiglu", 300, 520, 200),
                                        ("downproj", 520, 1000, 264)])
def test_stored_outputs_are_bit_identical_across_runs(name, M, N, K, variant):
    """The stored tensors do not depend on timing: five runs give the same
    bits (reductions, whose atomics may add in any order, are not compared).
    A race in the store path that moved a value by one ulp would pass the
    tolerance checks but not this one."""
    w = small(name, M, N, K)
    inp = synth.make_inputs(w, DEV)
    first = None
    for _ in range(5):
        plan, out = run_cuda(w, inp, debug_flags=VARIANTS[variant])
        got = (out.C.view(torch.int16).clone(), None if out.C8 is None else out.C8.clone())
        if first is None:
            first = got
        else:
            assert torch.equal(got[0], first[0])
            assert (got[1] is None) or torch.equal(got[1], first[1])


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("g,layout", [(2, "kn"), (4, "nk"), (8, "kn"), (16, "nk")])
def test_dswiglu_groups_and_ops(g, layout, variant):
    """The SwiGLU backward with every group, ops on dh before it (alpha, row
    scale) and on the 2N outputs after it (bias, AMAX, store, column sums)."""
    M, N, K = 260, 528, 136
    gen = torch.Generator(device=DEV).manual_seed(70 + g)
    A = torch.randn(M, K, generator=gen, device=DEV).to(torch.bfloat16)
    B = (torch.randn(*((K, N) if layout == "kn" else (N, K)), generator=gen, device=DEV) * 0.1).to(torch.bfloat16)
    pre = (torch.randn(M, 2 * N, generator=gen, device=DEV) * 1.5).to(torch.bfloat16)
    rs = torch.rand(M, generator=gen, device=DEV) + 0.5
    bias = torch.randn(2 * N, generator=gen, device=DEV) * 0.1
    prog = ["alpha", "row_scale", "dswiglu:%d" % g, "bias", "amax", "store_bf16", "col_sum"]
    plan = api.Plan(M, N, K, prog, b_layout=layout)
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, alpha=0.5, row_scale=rs, bias=bias, aux=pre, debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    p = oracle.Problem(bits(A), bits(B), prog, b_is_nk=(layout == "nk"), alpha=0.5, row_scale=rs.cpu().numpy(),
                       bias=bias.cpu().numpy(), preact=bits(pre))
    r = p.rows()
    check_bf16(bits(out.C), r["y"])
    check_amax(float(out.amax.item()), r["amax"])
    c = p.cols(list(range(2 * N)))
    check_cols(out.col_out.cpu().numpy(), c["col_stat"], np.abs(c["y"]).sum(0))


def test_two_library_copies_in_one_process(tmp_path):
    """A second copy of the library, loaded beside the first, launches its
    own kernels (each copy keeps its own kernel tables)."""
    import shutil
    copy = str(tmp_path / "libgemm_epi_copy.so")
    shutil.copy(native.LIB_PATH, copy)
    first = native.load()
    M, N, K = 200, 264, 128
    gen = torch.Generator(device=DEV).manual_seed(80)
    A = torch.randn(M, K, generator=gen, device=DEV).to(torch.bfloat16)
    B = torch.randn(K, N, generator=gen, device=DEV).to(torch.bfloat16)
    ref = oracle.Problem(bits(A), bits(B), ["gelu_tanh", "store_bf16"]).rows()["y"]
    results = []
    try:
        for lib_path in (native.LIB_PATH, copy, native.LIB_PATH):
            native._lib = first if lib_path == native.LIB_PATH else native.load(copy)
            plan = api.Plan(M, N, K, ["gelu_tanh", "store_bf16"])
            out = api.allocate_outputs(plan, DEV)
            api.run_program(plan, A, B, out)
            torch.cuda.synchronize()
            assert plan.query_status(out.workspace) == 0
            results.append(bits(out.C))
    finally:
        native._lib = first
    for r in results:
        check_bf16(r, ref)


# ------------------------------------------------------------ edge cases of the wider ops

@pytest.mark.parametrize("variant", ["1sm", "interp"])
def test_zero_k_backward_ops(variant):
    """K == 0: the accumulator is zero, so DSWIGLU gives the post-op bias
    alone and ROW_DOT gives zero sums, without reading A or B."""
    M, N = 130, 272
    gen = torch.Generator(device=DEV).manual_seed(90)
    A = torch.empty(M, 0, dtype=torch.bfloat16, device=DEV)
    B = torch.empty(0, N, dtype=torch.bfloat16, device=DEV)
    pre = torch.randn(M, 2 * N, generator=gen, device=DEV).to(torch.bfloat16)
    bias = torch.randn(2 * N, generator=gen, device=DEV)
    plan = api.Plan(M, N, 0, ["dswiglu", "bias", "store_bf16"])
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, aux=pre, bias=bias, debug_flags=VARIANTS[variant])
    x = torch.randn(M, N, generator=gen, device=DEV).to(torch.bfloat16)
    cs = torch.rand(N, generator=gen, device=DEV) + 0.5
    plan2 = api.Plan(M, N, 0, ["store_bf16", "col_scale", "row_dot"])
    out2 = api.allocate_outputs(plan2, DEV)
    out2.row_out.fill_(5.0)
    api.run_program(plan2, A, B, out2, aux=x, col_scale=cs, debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0 and plan2.query_status(out2.workspace) == 0
    check_bf16(bits(out.C), np.broadcast_to(bias.cpu().numpy().astype(np.float64), (M, 2 * N)))
    assert torch.all(out2.C.float() == 0) and torch.all(out2.row_out == 0)


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
def test_batched_two_weight_swiglu(variant):
    """Batches with separate gate / up weights (B and B2 advance together)."""
    Bt, M, N, K = 2, 200, 512, 136
    gen = torch.Generator(device=DEV).manual_seed(91)
    A = (torch.randn(Bt, M, K, generator=gen, device=DEV) * 0.5).to(torch.bfloat16)
    B = (torch.randn(Bt, K, N // 2, generator=gen, device=DEV) * 0.1).to(torch.bfloat16)
    B2 = (torch.randn(Bt, K, N // 2, generator=gen, device=DEV) * 0.1).to(torch.bfloat16)
    prog = ["pair_swiglu:128", "store_bf16"]
    plan = api.Plan(M, N, K, prog, dual=True, batch=Bt)
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, B2=B2, debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    for b in range(Bt):
        r = oracle.Problem(bits(A[b]), bits(B[b]), prog, B2=bits(B2[b])).rows()
        check_bf16(bits(out.C[b]), r["y"], "C[%d]" % b)


def test_rmsnorm_backward_empty_shapes():
    """M == 0 or N == 0 launches nothing; dw is still overwritten with zeros."""
    dw = torch.full((16,), 3.0, device=DEV)
    empty = torch.empty(0, 16, dtype=torch.bfloat16, device=DEV)
    s = torch.empty(0, device=DEV)
    api.rmsnorm_backward(empty, empty, s, s, dx=empty, dw=dw)
    none = torch.empty(4, 0, dtype=torch.bfloat16, device=DEV)
    api.rmsnorm_backward(none, none, torch.ones(4, device=DEV), torch.ones(4, device=DEV), dx=none)
    torch.cuda.synchronize()
    assert torch.all(dw == 0)


COMMON_PROGRAMS = [
    ["bias", "store_bf16"], ["bias", "gelu_tanh", "store_bf16"], ["bias", "relu", "store_bf16"],
    ["bias", "silu", "store_bf16"], ["alpha", "bias", "gelu_tanh", "store_bf16"], ["residual", "store_bf16"],
    ["gelu_tanh_grad", "store_bf16"], ["alpha", "store_bf16"], ["row_scale", "store_bf16"],
]


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("program", COMMON_PROGRAMS, ids=lambda p: ",".join(p))
def test_common_static_programs(program, variant):
    """The common programs compiled as static kernels (and, for comparison,
    through the interpreter) against the oracle."""
    M, N, K = 300, 528, 200
    gen = torch.Generator(device=DEV).manual_seed(130)
    A = (torch.randn(M, K, generator=gen, device=DEV) * 0.3).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=gen, device=DEV) * 0.3).to(torch.bfloat16)
    bias = torch.randn(N, generator=gen, device=DEV) * 0.2
    rs = torch.rand(M, generator=gen, device=DEV) + 0.5
    aux = torch.randn(M, N, generator=gen, device=DEV).to(torch.bfloat16)
    plan = api.Plan(M, N, K, program, b_layout="nk")
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, alpha=1.25, bias=bias, row_scale=rs, aux=aux, debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    r = oracle.Problem(bits(A), bits(B), program, b_is_nk=True, alpha=1.25, bias=bias.cpu().numpy(),
                       row_scale=rs.cpu().numpy(), residual=bits(aux) if "residual" in program else None,
                       preact=bits(aux) if "gelu_tanh_grad" in program else None).rows()
    check_bf16(bits(out.C), r["y"])
