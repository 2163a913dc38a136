"""The C-ABI library without a GPU: it loads, exports every entry point that
include/gemm_epi.h declares, and validates descriptors on the host
(gemm_epi_create does no CUDA call).  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

from gemm_epilogue_transformer_smem_gb300 import api, build, native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_epi.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return N.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_epi_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", N.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (gemm_epi_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    # the binding covers the same set
    assert set(names) == {s[0] for s in N.SIGNATURES}


def test_only_the_c_abi_is_exported(lib):
    """Hidden visibility: the library exports exactly the declared entry
    points and no GNU-unique symbols, which the loader would otherwise merge
    across two copies of the library in one process."""
    out = subprocess.run(["nm", "-D", "--defined-only", N.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    defined = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert defined == set(declared_functions()), sorted(defined ^ set(declared_functions()))
    assert not any(line.split()[1] == "u" for line in out.splitlines() if len(line.split()) >= 3)


def test_struct_layouts_match_header(lib, tmp_path):
    """Size and every field offset of the three structs, as a C compiler lays
    them out from the header, against the ctypes binding."""
    structs = [N.gemm_epi_op, N.gemm_epi_desc, N.gemm_epi_args]
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "gemm_epi.h"', "int main(void) {"]
    for st in structs:
        name = st.__name__
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (name, name))
        for f, _ in st._fields_:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (name, f, name, f))
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for st in structs:
        name = st.__name__
        assert int(got[name]) == ctypes.sizeof(st), name
        for f, _ in st._fields_:
            assert int(got["%s.%s" % (name, f)]) == getattr(st, f).offset, (name, f)


def test_version_and_status_strings(lib):
    assert lib.gemm_epi_version() == 1
    for code in range(8):
        assert lib.gemm_epi_status_string(code)
    assert lib.gemm_epi_status_string(99) == b"unknown status"


def create(lib, M=256, N_=512, K=128, program=("store_bf16",), layout=N.GEMM_EPI_B_KN, **strides):
    ops = api.encode_program(list(program))
    d = N.gemm_epi_desc()
    d.M, d.N, d.K = M, N_, K
    n_out = api.out_cols(list(program), N_)
    d.lda = strides.get("lda", K)
    d.ldb = strides.get("ldb", N_ if layout == N.GEMM_EPI_B_KN else K)
    d.ldc = strides.get("ldc", n_out)
    d.ldc8 = strides.get("ldc8", n_out)
    d.ld_aux = strides.get("ld_aux", n_out)
    d.b_layout = layout
    d.a_type, d.b_type = strides.get("a_type", 0), strides.get("b_type", 0)
    d.n_ops = strides.get("n_ops", len(program))
    d.ops = ctypes.cast(ops, ctypes.POINTER(N.gemm_epi_op))
    h = N.gemm_epi_handle()
    s = lib.gemm_epi_create(ctypes.byref(h), ctypes.byref(d))
    return s, h


@pytest.mark.parametrize("program", [
    ("store_bf16",),
    ("alpha", "bias", "gelu_tanh", "amax", "store_bf16"),
    ("pair_swiglu", "store_bf16"),
    ("alpha", "bias", "relu", "amax", "store_bf16", "store_e4m3"),
    ("residual", "store_bf16", "row_rms:1e-6"),
    ("gelu_tanh_grad", "store_bf16", "col_sum"),
    (),
])
def test_create_accepts_programs(lib, program):
    s, h = create(lib, program=program)
    assert s == N.GEMM_EPI_OK, lib.gemm_epi_last_error()
    pair = any(p.startswith("pair") for p in program)
    assert lib.gemm_epi_out_cols(h) == (256 if pair else 512)
    ws = lib.gemm_epi_workspace_size(h)
    assert ws >= 256 and ws % 256 == 0
    assert lib.gemm_epi_destroy(h) == N.GEMM_EPI_OK


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_create_accepts_dswiglu(lib, g):
    prog = ("alpha", "row_scale", "dswiglu:%d" % g, "bias", "amax", "store_bf16", "col_sum")
    s, h = create(lib, program=prog, ld_aux=1024)
    assert s == N.GEMM_EPI_OK, lib.gemm_epi_last_error()
    assert lib.gemm_epi_out_cols(h) == 1024
    assert lib.gemm_epi_destroy(h) == N.GEMM_EPI_OK
    assert api.out_cols(list(prog), 512) == 1024


@pytest.mark.parametrize("types", [(1, 1), (1, 2), (2, 1), (2, 2)])
def test_create_accepts_fp8_operands(lib, types):
    s, h = create(lib, layout=N.GEMM_EPI_B_NK, a_type=types[0], b_type=types[1], K=144, lda=160, ldb=176,
                  program=("alpha", "bias", "relu", "amax", "store_bf16", "store_e4m3"))
    assert s == N.GEMM_EPI_OK, lib.gemm_epi_last_error()
    assert lib.gemm_epi_destroy(h) == N.GEMM_EPI_OK


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(K=2 ** 31), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(layout=7), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(lda=64), N.GEMM_EPI_ERR_INVALID_VALUE),          # lda < K
    (dict(lda=132), N.GEMM_EPI_ERR_MISALIGNED),            # not a multiple of 8
    (dict(K=12, lda=16), N.GEMM_EPI_ERR_MISALIGNED),       # K tail inside a 16-byte group
    (dict(ldb=516), N.GEMM_EPI_ERR_MISALIGNED),
    (dict(ldc=500), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(ldc=516), N.GEMM_EPI_ERR_MISALIGNED),
    (dict(program=("store_bf16", "store_e4m3"), ldc8=520), N.GEMM_EPI_ERR_MISALIGNED),
    (dict(program=("store_bf16", "store_bf16")), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("store_bf16", "row_dot", "row_dot"), ld_aux=512), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("store_bf16", "row_rms", "row_dot"), ld_aux=512), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("col_sum", "col_sum")), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("pair_swiglu", "pair_swiglu")), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("pair_swiglu:3", "store_bf16")), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(N_=511, program=("pair_swiglu", "store_bf16")), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(N_=520, program=("pair_swiglu:8", "store_bf16")), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("residual", "pair_swiglu", "store_bf16")), N.GEMM_EPI_ERR_UNSUPPORTED),
    (dict(program=("store_bf16", "pair_swiglu")), N.GEMM_EPI_ERR_UNSUPPORTED),
    (dict(program=("residual", "gelu_tanh_grad", "store_bf16")), N.GEMM_EPI_ERR_UNSUPPORTED),
    (dict(program=("residual", "store_bf16"), ld_aux=12), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(N_=0, program=("row_rms",)), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("store_bf16",), n_ops=17), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(layout=N.GEMM_EPI_B_KN | N.GEMM_EPI_B_DUAL, N_=384, program=("pair_swiglu:128", "store_bf16"),
          ldb=192), N.GEMM_EPI_ERR_INVALID_VALUE),                       # N % 256
    (dict(layout=N.GEMM_EPI_B_KN | N.GEMM_EPI_B_DUAL, program=("pair_swiglu", "store_bf16"), ldb=256),
     N.GEMM_EPI_ERR_INVALID_VALUE),                                      # group must be 128
    (dict(program=("bias", "pair_swiglu:128", "store_bf16")), N.GEMM_EPI_ERR_UNSUPPORTED),
    (dict(layout=N.GEMM_EPI_B_NK | 32, program=("store_bf16",)), N.GEMM_EPI_ERR_INVALID_VALUE),
    # SwiGLU backward
    (dict(program=("dswiglu:32", "store_bf16"), ld_aux=1024), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(N_=500, program=("dswiglu:8", "store_bf16"), ld_aux=1024), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("dswiglu", "residual", "store_bf16"), ld_aux=1024), N.GEMM_EPI_ERR_UNSUPPORTED),
    (dict(program=("dswiglu", "gelu_tanh_grad", "store_bf16"), ld_aux=1024), N.GEMM_EPI_ERR_UNSUPPORTED),
    (dict(program=("dswiglu", "pair_swiglu", "store_bf16"), ld_aux=1024), N.GEMM_EPI_ERR_INVALID_VALUE),
    (dict(program=("store_bf16", "dswiglu"), ld_aux=1024), N.GEMM_EPI_ERR_UNSUPPORTED),
    (dict(program=("dswiglu", "store_bf16"), ld_aux=1000), N.GEMM_EPI_ERR_INVALID_VALUE),  # ld_aux < 2N
    (dict(layout=N.GEMM_EPI_B_KN | N.GEMM_EPI_B_DUAL, program=("dswiglu", "store_bf16"), ldb=256, ld_aux=1024),
     N.GEMM_EPI_ERR_UNSUPPORTED),
    # 8-bit operands
    (dict(a_type=3), N.GEMM_EPI_ERR_INVALID_VALUE),                      # unknown type
    (dict(layout=N.GEMM_EPI_B_NK, a_type=1), N.GEMM_EPI_ERR_UNSUPPORTED),  # FP8 A with bf16 B
    (dict(layout=N.GEMM_EPI_B_NK, b_type=2), N.GEMM_EPI_ERR_UNSUPPORTED),  # bf16 A with FP8 B
    (dict(a_type=1, b_type=1), N.GEMM_EPI_ERR_UNSUPPORTED),             # FP8 needs B stored N x K
    (dict(layout=N.GEMM_EPI_B_NK, a_type=1, b_type=1, K=136, lda=144, ldb=144), N.GEMM_EPI_ERR_MISALIGNED),
    (dict(layout=N.GEMM_EPI_B_NK, a_type=1, b_type=1, lda=136), N.GEMM_EPI_ERR_MISALIGNED),
    (dict(layout=N.GEMM_EPI_B_NK, a_type=2, b_type=1, ldb=136), N.GEMM_EPI_ERR_MISALIGNED),
])

def test_create_rejects(lib, kw, status):
    s, h = create(lib, **kw)
    assert s == status, (s, lib.gemm_epi_last_error())
    assert lib.gemm_epi_last_error()
    assert not h.value


def test_create_rejects_unknown_op_and_nulls(lib):
    bad = (N.gemm_epi_op * 1)(N.gemm_epi_op(99, 0, 0.0))
    d = N.gemm_epi_desc(M=8, N=8, K=8, lda=8, ldb=8, ldc=8, ldc8=16, ld_aux=8, b_layout=0, n_ops=1,
                        ops=ctypes.cast(bad, ctypes.POINTER(N.gemm_epi_op)))
    h = N.gemm_epi_handle()
    assert lib.gemm_epi_create(ctypes.byref(h), ctypes.byref(d)) == N.GEMM_EPI_ERR_INVALID_VALUE
    assert lib.gemm_epi_create(None, ctypes.byref(d)) == N.GEMM_EPI_ERR_INVALID_VALUE
    assert lib.gemm_epi_create(ctypes.byref(h), None) == N.GEMM_EPI_ERR_INVALID_VALUE
    d.n_ops, d.ops = 2, None
    assert lib.gemm_epi_create(ctypes.byref(h), ctypes.byref(d)) == N.GEMM_EPI_ERR_INVALID_VALUE
    assert lib.gemm_epi_destroy(None) == N.GEMM_EPI_OK
    assert lib.gemm_epi_workspace_size(None) == 0
    assert lib.gemm_epi_out_cols(None) == -1


def test_zero_k_needs_no_operand_strides(lib):
    s, h = create(lib, K=0, lda=0, program=("bias", "store_bf16"))
    assert s == N.GEMM_EPI_OK, lib.gemm_epi_last_error()
    lib.gemm_epi_destroy(h)


def test_workspace_grows_with_row_tiles(lib):
    s1, h1 = create(lib, M=128, program=("residual", "store_bf16", "row_rms"))
    s2, h2 = create(lib, M=128 * 200, program=("residual", "store_bf16", "row_rms"))
    assert s1 == s2 == N.GEMM_EPI_OK
    assert lib.gemm_epi_workspace_size(h2) >= 256 + 4 * 200 > lib.gemm_epi_workspace_size(h1) - 1
    lib.gemm_epi_destroy(h1)
    lib.gemm_epi_destroy(h2)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        N.load(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("layout", [N.GEMM_EPI_B_KN, N.GEMM_EPI_B_NK])
def test_create_accepts_two_weight_programs(lib, layout):
    for prog in (("pair_swiglu:128", "store_bf16"), ("row_scale", "pair_mul:128", "store_bf16"),
                 ("store_bf16",)):
        s, h = create(lib, N_=512, program=prog, layout=layout | N.GEMM_EPI_B_DUAL,
                      ldb=256 if layout == N.GEMM_EPI_B_KN else 128)
        assert s == N.GEMM_EPI_OK, lib.gemm_epi_last_error()
        pair = any(p.startswith("pair") for p in prog)
        assert lib.gemm_epi_out_cols(h) == (256 if pair else 512)
        lib.gemm_epi_destroy(h)


def test_create_checks_batch_strides(lib):
    def desc(**kw):
        ops = api.encode_program(["residual", "store_bf16", "row_rms"])
        d = N.gemm_epi_desc(M=256, N=512, K=128, lda=128, ldb=512, ldc=512, ldc8=512, ld_aux=512,
                            b_layout=N.GEMM_EPI_B_KN, n_ops=3, ops=ctypes.cast(ops, ctypes.POINTER(N.gemm_epi_op)))
        d.batch, d.batch_stride_a, d.batch_stride_b = 4, 256 * 128, 128 * 512
        d.batch_stride_c, d.batch_stride_aux = 256 * 512, 256 * 512
        for k, v in kw.items():
            setattr(d, k, v)
        h = N.gemm_epi_handle()
        return lib.gemm_epi_create(ctypes.byref(h), ctypes.byref(d)), h, ops
    s, h, _ = desc()
    assert s == N.GEMM_EPI_OK, lib.gemm_epi_last_error()
    one, h1, _ = desc(batch=1)
    # one row counter per 128-row block of every batch
    assert lib.gemm_epi_workspace_size(h) >= 256 + 4 * 2 * 4
    assert lib.gemm_epi_workspace_size(h) >= lib.gemm_epi_workspace_size(h1)
    lib.gemm_epi_destroy(h)
    lib.gemm_epi_destroy(h1)
    s, h, _ = desc(batch_stride_b=0)          # shared weights
    assert s == N.GEMM_EPI_OK
    lib.gemm_epi_destroy(h)
    for bad in (dict(batch_stride_c=0), dict(batch_stride_c=512), dict(batch_stride_a=100),
                dict(batch_stride_aux=256 * 512 - 8), dict(batch=-1), dict(batch=70000)):
        s, h, _ = desc(**bad)
        assert s == N.GEMM_EPI_ERR_INVALID_VALUE, bad


@pytest.mark.parametrize("name", sorted(__import__("gemm_epilogue_transformer_smem_gb300.synth",
                                                   fromlist=["WORKLOADS"]).WORKLOADS))
def test_binding_supplies_every_argument_a_workload_needs(lib, name):
    """Each workload's program through the Python binding with host tensors:
    every pointer the program uses is present and aligned, so the call gets
    past the argument checks and stops only at the missing GPU."""
    import torch
    from gemm_epilogue_transformer_smem_gb300 import synth
    w = synth.WORKLOADS[name]
    w = w.scaled(min(w.M, 96), min(w.N, 512), min(w.K, 128))
    inp = synth.make_inputs(w, "cpu")
    plan = api.Plan(w.M, w.N, w.K, w.program, b_layout=w.b_layout, dual=w.dual, a_type=w.in_type,
                    b_type=w.in_type, batch=w.batch)
    out = api.allocate_outputs(plan, "cpu")
    with pytest.raises(N.GemmEpiError) as err:
        api.run_program(plan, inp.A, inp.B, out, alpha=inp.alpha, fp8_scale=inp.fp8_scale, bias=inp.bias,
                        aux=inp.aux, B2=inp.B2, a_scale_inv=inp.a_scale_inv, b_scale_inv=inp.b_scale_inv,
                        col_scale=inp.col_scale, row_scale=inp.row_scale, stream=FakeStream())
    assert err.value.status in (N.GEMM_EPI_ERR_CUDA, N.GEMM_EPI_ERR_ARCH), str(err.value)
    if w.finish == "rmsnorm_backward":
        dx = torch.empty(out.C.shape, dtype=torch.bfloat16)
        dw = torch.empty(out.C.shape[1])
        with pytest.raises(N.GemmEpiError) as err:
            api.rmsnorm_backward(out.C, inp.aux, inp.row_stat, out.row_out, w=inp.col_scale, dx=dx, dw=dw,
                                 stream=FakeStream())
        assert err.value.status in (N.GEMM_EPI_ERR_CUDA, N.GEMM_EPI_ERR_ARCH), str(err.value)


class FakeStream:
    """Stands in for a torch CUDA stream on a machine without a GPU."""
    cuda_stream = 0


def test_rmsnorm_backward_checks_arguments_on_the_host(lib):
    """gemm_epi_rmsnorm_backward validates every pointer and stride before it
    touches the device, so these errors come back without a GPU."""
    M, N_ = 8, 16
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256  # 16-byte aligned, never dereferenced on the host

    def args(**kw):
        a = N.gemm_epi_rmsnorm_bwd_args()
        a.M, a.N = M, N_
        a.dy, a.ld_dy, a.x, a.ld_x = base, N_, base, N_
        a.s, a.r, a.dx, a.ld_dx = base, base, base, N_
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    cases = [
        (dict(dy=None), N.GEMM_EPI_ERR_INVALID_VALUE),           # dy is NULL
        (dict(dy=base + 2), N.GEMM_EPI_ERR_MISALIGNED),          # dy not 16-byte aligned
        (dict(ld_x=N_ - 8), N.GEMM_EPI_ERR_INVALID_VALUE),       # row stride < N
        (dict(ld_dx=N_ + 4), N.GEMM_EPI_ERR_MISALIGNED),         # stride not a multiple of 8
        (dict(r=None), N.GEMM_EPI_ERR_INVALID_VALUE),            # dx needs r
        (dict(s=base + 2), N.GEMM_EPI_ERR_MISALIGNED),           # fp32 vectors 4-byte aligned
        (dict(dw=base + 2), N.GEMM_EPI_ERR_MISALIGNED),
        (dict(M=-1), N.GEMM_EPI_ERR_INVALID_VALUE),
    ]
    for kw, status in cases:
        a = args(**kw)
        assert lib.gemm_epi_rmsnorm_backward(ctypes.byref(a), None) == status, kw
    assert lib.gemm_epi_rmsnorm_backward(None, None) == N.GEMM_EPI_ERR_INVALID_VALUE


def test_binding_checks_dtypes_and_extents(lib):
    """The C ABI sees only pointers, so the binding checks each tensor's
    dtype and that its storage covers the declared extent before the call."""
    import torch
    M, N_, K = 64, 256, 128
    plan = api.Plan(M, N_, K, ["bias", "pair_swiglu", "store_bf16", "amax"])
    A = torch.zeros(M, K, dtype=torch.bfloat16)
    B = torch.zeros(K, N_, dtype=torch.bfloat16)
    C = torch.zeros(M, N_ // 2, dtype=torch.bfloat16)
    amax = torch.zeros(1)
    bias = torch.zeros(N_)  # before the pair op: N values
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8)
    ok = dict(bias=bias, C=C, amax=amax, workspace=ws)
    plan.args(A, B, **ok)
    with pytest.raises(TypeError, match="A: expected a bf16"):
        plan.args(A.float(), B, **ok)
    with pytest.raises(TypeError, match="amax"):
        plan.args(A, B, **dict(ok, amax=torch.zeros(1, dtype=torch.float64)))
    with pytest.raises(ValueError, match="C: "):
        plan.args(A, B, **dict(ok, C=C[1:]))          # one row short
    with pytest.raises(ValueError, match="B: "):
        plan.args(A, B.reshape(-1)[: K * N_ - 1].clone(), **ok)  # one element short
    plan.args(A, B.reshape(-1).clone(), **ok)        # any shape whose storage covers K x N
    plan.args(A, B[:, :8], **ok)                     # a view: its storage covers K x N
    with pytest.raises(ValueError, match="bias"):
        plan.args(A, B, **dict(ok, bias=bias[: N_ // 2].clone()))
    # 8-bit operands accept any one-byte dtype; batched extents count every problem
    p8 = api.Plan(M, N_, K, ["store_bf16"], b_layout="nk", a_type="e4m3", b_type="e4m3", batch=3,
                  batch_stride_b=0)
    A8, B8 = torch.zeros(3, M, K, dtype=torch.uint8), torch.zeros(N_, K, dtype=torch.float8_e4m3fn)
    C3 = torch.zeros(3, M, N_, dtype=torch.bfloat16)
    p8.args(A8, B8, C=C3, workspace=ws)
    with pytest.raises(ValueError, match="A: "):
        p8.args(A8[:2].clone(), B8, C=C3, workspace=ws)
    with pytest.raises(TypeError, match="B: expected a byte"):
        p8.args(A8, B8.to(torch.bfloat16), C=C3, workspace=ws)


def test_rmsnorm_backward_binding_checks(lib):
    import torch
    M, N_ = 16, 64
    dy, x = torch.zeros(M, N_, dtype=torch.bfloat16), torch.zeros(M, N_, dtype=torch.bfloat16)
    s, r = torch.ones(M), torch.ones(M)
    with pytest.raises(TypeError, match="dy"):
        api.rmsnorm_backward(dy.float(), x, s, r, dx=x)
    with pytest.raises(TypeError, match="r: "):
        api.rmsnorm_backward(dy, x, s, r.double(), dx=x)
    with pytest.raises(ValueError, match="w: "):
        api.rmsnorm_backward(dy, x, s, r, w=torch.ones(N_ - 1), dx=x)
    with pytest.raises(ValueError, match="dx: "):
        api.rmsnorm_backward(dy, x, s, r, dx=x[1:].reshape(M - 1, N_))
