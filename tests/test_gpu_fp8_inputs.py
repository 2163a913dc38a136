"""GEMMs on FP8 operands (tcgen05 kind::f8f6f4) against the oracle, through
the C ABI (needs a GB300).

The FP8 loop of the cuDNN Graph API tutorial's matmul epilogue paragraph:
one GEMM's epilogue quantises its output with a scale fixed by an expected
AMAX and reports the AMAX; the next GEMM reads those e4m3 codes and
multiplies its accumulator by the reciprocal scale, read from device memory.
Both e4m3 and e5m2 operands, the dequantisation factors present or absent,
two weight operands, batches, and the two-stage chain.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_epilogue_transformer_smem_gb300 import api, native

from parity import bits, check_amax, check_bf16, check_e4m3

pytestmark = pytest.mark.gpu

DEV = "cuda"
FMT = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
VARIANTS = {"1sm": native.GEMM_EPI_DEBUG_FORCE_1SM, "2sm": native.GEMM_EPI_DEBUG_FORCE_2SM,
            "interp": native.GEMM_EPI_DEBUG_FORCE_INTERPRETER}


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    assert torch.cuda.is_available()
    return cuda_lib


def codes(shape, fmt, scale, g, relu=False):
    t = torch.randn(*shape, generator=g, device=DEV)
    if relu:
        t.clamp_min_(0)
    lim = torch.finfo(FMT[fmt]).max
    return (t * scale).clamp_(-lim, lim).to(FMT[fmt]).view(torch.uint8)


def dev_scalar(x):
    return torch.tensor([x], dtype=torch.float32, device=DEV)


def host(t):
    return t.contiguous().cpu().numpy()


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("a_t,b_t", [("e4m3", "e5m2"), ("e5m2", "e4m3"), ("e5m2", "e5m2")])
def test_operand_type_mixes(a_t, b_t, variant):
    M, N, K = 300, 520, 400  # ragged M, N; K = 3 blocks of 128 + 16
    g = torch.Generator(device=DEV).manual_seed(31)
    A = codes((M, K), a_t, 24.0, g)
    B = codes((N, K), b_t, 24.0, g)
    sa, sb = 1.0 / 24.0, 1.0 / (24.0 * K ** 0.5)
    prog = ["alpha", "gelu_tanh", "amax", "store_bf16"]
    plan = api.Plan(M, N, K, prog, b_layout="nk", a_type=a_t, b_type=b_t)
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, alpha=1.5, a_scale_inv=dev_scalar(sa), b_scale_inv=dev_scalar(sb),
                    debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    r = oracle.Problem(host(A), host(B), prog, b_is_nk=True, alpha=1.5, a_type=a_t, b_type=b_t,
                       a_scale_inv=sa, b_scale_inv=sb).rows()
    check_bf16(bits(out.C), r["y"])
    check_amax(float(out.amax.item()), r["amax"])


@pytest.mark.parametrize("which", ["none", "a", "b", "both"])
def test_dequantisation_factors(which):
    """Each factor applies on its own, NULL means 1, and a missing factor is
    not silently taken from the other operand (distinct values)."""
    M, N, K = 256, 256, 256
    g = torch.Generator(device=DEV).manual_seed(32)
    A = codes((M, K), "e4m3", 16.0, g)
    B = codes((N, K), "e4m3", 16.0, g)
    sa = 0.0625 if which in ("a", "both") else None
    sb = 0.0078125 if which in ("b", "both") else None
    plan = api.Plan(M, N, K, ["store_bf16"], b_layout="nk", a_type="e4m3", b_type="e4m3")
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, a_scale_inv=None if sa is None else dev_scalar(sa),
                    b_scale_inv=None if sb is None else dev_scalar(sb))
    torch.cuda.synchronize()
    r = oracle.Problem(host(A), host(B), ["store_bf16"], b_is_nk=True, a_type="e4m3", b_type="e4m3",
                       a_scale_inv=sa or 1.0, b_scale_inv=sb or 1.0).rows()
    check_bf16(bits(out.C), r["y"])


def test_dequantisation_factor_on_bf16_operands():
    """The factors are not tied to FP8: a bf16 GEMM scaled by them."""
    M, N, K = 200, 264, 128
    g = torch.Generator(device=DEV).manual_seed(33)
    A = torch.randn(M, K, generator=g, device=DEV).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g, device=DEV).to(torch.bfloat16)
    plan = api.Plan(M, N, K, ["store_bf16"])
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, a_scale_inv=dev_scalar(0.25), b_scale_inv=dev_scalar(3.0))
    torch.cuda.synchronize()
    r = oracle.Problem(bits(A), bits(B), ["store_bf16"], a_scale_inv=0.25, b_scale_inv=3.0).rows()
    check_bf16(bits(out.C), r["y"])


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
def test_two_weight_fp8(variant):
    M, N, K = 300, 768, 256
    g = torch.Generator(device=DEV).manual_seed(34)
    A = codes((M, K), "e4m3", 32.0, g, relu=True)
    B = codes((N // 2, K), "e4m3", 32.0, g)
    B2 = codes((N // 2, K), "e4m3", 32.0, g)
    sa, sb = 1.0 / 32.0, 1.0 / (32.0 * K ** 0.5)
    prog = ["pair_swiglu:128", "store_bf16"]
    plan = api.Plan(M, N, K, prog, b_layout="nk", dual=True, a_type="e4m3", b_type="e4m3")
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, B2=B2, a_scale_inv=dev_scalar(sa), b_scale_inv=dev_scalar(sb),
                    debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    r = oracle.Problem(host(A), host(B), prog, b_is_nk=True, B2=host(B2), a_type="e4m3", b_type="e4m3",
                       a_scale_inv=sa, b_scale_inv=sb).rows()
    check_bf16(bits(out.C), r["y"])


@pytest.mark.parametrize("shared_b", [False, True])
def test_batched_fp8(shared_b):
    Bt, M, N, K = 3, 160, 272, 192
    g = torch.Generator(device=DEV).manual_seed(35)
    A = codes((Bt, M, K), "e4m3", 32.0, g)
    B = codes((N, K) if shared_b else (Bt, N, K), "e4m3", 32.0, g)
    sa, sb = 1.0 / 32.0, 1.0 / 256.0
    prog = ["amax", "store_bf16", "store_e4m3"]
    plan = api.Plan(M, N, K, prog, b_layout="nk", batch=Bt, batch_stride_b=0 if shared_b else None,
                    a_type="e4m3", b_type="e4m3")
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, fp8_scale=16.0, a_scale_inv=dev_scalar(sa), b_scale_inv=dev_scalar(sb))
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    amax = 0.0
    for b in range(Bt):
        r = oracle.Problem(host(A[b]), host(B if shared_b else B[b]), prog, b_is_nk=True, fp8_scale=16.0,
                           a_type="e4m3", b_type="e4m3", a_scale_inv=sa, b_scale_inv=sb).rows()
        check_bf16(bits(out.C[b]), r["y"], "C[%d]" % b)
        check_e4m3(host(out.C8[b]), r["c_e4m3"], r["y"] * 16.0)
        amax = max(amax, r["amax"])
    check_amax(float(out.amax.item()), amax)


def test_fp8_loop_chain():
    """Stage 1 is the fp8 workload's program (relu(0.5 acc + bias), AMAX,
    e4m3 at scale 448/4); stage 2 reads stage 1's e4m3 codes as A with the
    reciprocal scale from device memory and an e4m3 weight.  The stage-2
    oracle reads the oracle's own stage-1 codes, never the GPU's."""
    M, K1, H, N2 = 384, 512, 768, 640
    g = torch.Generator(device=DEV).manual_seed(36)
    X = (torch.randn(M, K1, generator=g, device=DEV) / K1 ** 0.5).to(torch.bfloat16)
    W1 = (torch.randn(K1, H, generator=g, device=DEV) / K1 ** 0.5).to(torch.bfloat16)
    bias1 = torch.randn(H, generator=g, device=DEV) * 0.1
    qw = 112.0 * H ** 0.5
    W2 = codes((N2, H), "e4m3", 112.0, g)  # N(0, 1/sqrt(H)) weights at scale 112 sqrt(H)
    prog1 = ["alpha", "bias", "relu", "amax", "store_bf16", "store_e4m3"]
    prog2 = ["alpha", "gelu_tanh", "store_bf16"]
    p1 = api.Plan(M, H, K1, prog1)
    o1 = api.allocate_outputs(p1, DEV)
    api.run_program(p1, X, W1, o1, alpha=0.5, bias=bias1, fp8_scale=112.0)
    s1_inv = torch.full((1,), 1.0 / 112.0, dtype=torch.float32, device=DEV)
    p2 = api.Plan(M, N2, H, prog2, b_layout="nk", a_type="e4m3", b_type="e4m3")
    o2 = api.allocate_outputs(p2, DEV)
    api.run_program(p2, o1.C8, W2, o2, alpha=2.0, a_scale_inv=s1_inv, b_scale_inv=dev_scalar(1.0 / qw))
    torch.cuda.synchronize()
    assert p1.query_status(o1.workspace) == 0 and p2.query_status(o2.workspace) == 0

    r1 = oracle.Problem(bits(X), bits(W1), prog1, alpha=0.5, bias=host(bias1), fp8_scale=112.0).rows()
    check_e4m3(host(o1.C8), r1["c_e4m3"], r1["y"] * 112.0)
    check_amax(float(o1.amax.item()), r1["amax"])
    assert r1["amax"] * 112.0 <= 448.0  # the scale leaves the codes unsaturated
    W2h = host(W2)
    r2 = oracle.Problem(r1["c_e4m3"], W2h, prog2, b_is_nk=True, alpha=2.0, a_type="e4m3", b_type="e4m3",
                        a_scale_inv=float(np.float32(1.0 / 112.0)), b_scale_inv=float(np.float32(1.0 / qw))).rows()
    # Stage 1 may pick the other of two adjacent codes where its value lies
    # next to a midpoint (allowed above); carried through stage 2's GEMM,
    # alpha and gelu (|gelu'| <= 1.13) that bounds the extra difference.
    dA = np.abs(oracle.e4m3_to_f64(host(o1.C8)) - oracle.e4m3_to_f64(r1["c_e4m3"]))
    Wd = np.abs(oracle.e4m3_to_f64(W2h))
    prop = 1.13 * 2.0 * (dA @ Wd.T) / 112.0 / qw
    g2 = oracle.bf16_bits_to_f64(bits(o2.C))
    rms = float(np.sqrt(np.mean(r2["y"] ** 2)))
    bound = 2e-2 * np.maximum(np.abs(r2["y"]), 1e-2 * rms) + prop
    bad = np.abs(g2 - r2["y"]) > bound
    assert not bad.any(), "chain output: %d of %d outside the propagated bound" % (int(bad.sum()), bad.size)


@pytest.mark.parametrize("variant", ["1sm", "2sm"])
def test_fp8_backward_program(variant):
    """A backward GEMM of the FP8 loop: e5m2 gradients times e4m3 weights,
    finished by the SwiGLU backward epilogue."""
    M, N, K = 260, 272, 192
    g = torch.Generator(device=DEV).manual_seed(37)
    A = codes((M, K), "e5m2", 64.0, g)
    B = codes((N, K), "e4m3", 64.0, g)
    pre = (torch.randn(M, 2 * N, generator=g, device=DEV) * 1.3).to(torch.bfloat16)
    sa, sb = 1.0 / 64.0, 1.0 / (64.0 * K ** 0.5)
    prog = ["dswiglu", "amax", "store_bf16"]
    plan = api.Plan(M, N, K, prog, b_layout="nk", a_type="e5m2", b_type="e4m3")
    out = api.allocate_outputs(plan, DEV)
    api.run_program(plan, A, B, out, aux=pre, a_scale_inv=dev_scalar(sa), b_scale_inv=dev_scalar(sb),
                    debug_flags=VARIANTS[variant])
    torch.cuda.synchronize()
    assert plan.query_status(out.workspace) == 0
    r = oracle.Problem(host(A), host(B), prog, b_is_nk=True, preact=bits(pre), a_type="e5m2", b_type="e4m3",
                       a_scale_inv=sa, b_scale_inv=sb).rows()
    check_bf16(bits(out.C), r["y"])
    check_amax(float(out.amax.item()), r["amax"])
