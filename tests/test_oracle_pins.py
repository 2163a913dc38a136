"""Pins of the fp64 CPU oracle to things other than itself.

Each test checks the oracle against numpy, a closed form, an exact special
case, a hand-derived table or a pure-Python brute force, chosen so that a
plausible mistake (a dropped term, a wrong sign or index, a transposed
operand, swapped gate/up) fails at least one of them.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import Problem

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(7)


def bf16_bits_from_f32(x):
    """bf16 bit patterns via torch's own float32 -> bfloat16 conversion."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_bf16(shape, scale=1.0):
    return bf16_bits_from_f32(RNG.standard_normal(shape) * scale)


def f64(bits):
    return oracle.bf16_bits_to_f64(bits)


# ---------------------------------------------------------------- GEMM

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 33, 65), (64, 40, 24)])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_gemm_matches_numpy_einsum(M, N, K, layout):
    A = rand_bf16((M, K))
    B = rand_bf16((K, N) if layout == "kn" else (N, K))
    y = Problem(A, B, [], b_is_nk=(layout == "nk")).rows()["y"]
    Bk = f64(B) if layout == "kn" else f64(B).T
    ref = np.einsum("mk,kn->mn", f64(A), Bk)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_gemm_integer_exact():
    A = bf16_bits_from_f32(RNG.integers(-2, 3, (24, 40)))
    B = bf16_bits_from_f32(RNG.integers(-2, 3, (40, 16)))
    y = Problem(A, B, []).rows()["y"]
    ref = f64(A).astype(np.int64) @ f64(B).astype(np.int64)
    assert np.array_equal(y, ref.astype(np.float64))


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_identity_and_permutation(layout):
    K = 12
    B = rand_bf16((K, 9) if layout == "kn" else (9, K))
    Bkn = f64(B) if layout == "kn" else f64(B).T
    eye = bf16_bits_from_f32(np.eye(K))
    y = Problem(eye, B, [], b_is_nk=(layout == "nk")).rows()["y"]
    assert np.array_equal(y, Bkn)
    perm = RNG.permutation(K)
    P = bf16_bits_from_f32(np.eye(K)[perm])
    y = Problem(P, B, [], b_is_nk=(layout == "nk")).rows()["y"]
    assert np.array_equal(y, Bkn[perm])


def test_gemm_transposed_operand_is_caught():
    """Planted mistake: reading a K x N B as if it were N x K must not pass
    the einsum pin (square, non-symmetric B)."""
    A = rand_bf16((4, 8))
    B = rand_bf16((8, 8))
    wrong = Problem(A, B, [], b_is_nk=True).rows()["y"]
    ref = f64(A) @ f64(B)
    assert not np.allclose(wrong, ref, rtol=1e-6)


# ---------------------------------------------------------------- activations

def gelu_tanh_textbook(x):
    return 0.5 * x * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


@pytest.mark.parametrize("x", [-8.0, -3.0, -1.0, -0.75, -0.1, 0.0, 1e-3, 0.5, 1.0, 2.5, 6.0])
def test_gelu_tanh_closed_forms(x):
    g = oracle.gelu_tanh
    assert g(x) == pytest.approx(gelu_tanh_textbook(x), rel=1e-12, abs=1e-15)
    assert g(x) - g(-x) == pytest.approx(x, rel=1e-12, abs=1e-15)
    d = oracle.gelu_tanh_grad
    assert d(x) + d(-x) == pytest.approx(1.0, rel=1e-12)
    h = 1e-5
    fd = (gelu_tanh_textbook(x + h) - gelu_tanh_textbook(x - h)) / (2 * h)
    assert d(x) == pytest.approx(fd, rel=1e-7, abs=1e-9)


def test_gelu_special_values():
    assert oracle.gelu_tanh(0.0) == 0.0
    assert oracle.gelu_tanh_grad(0.0) == 0.5


@pytest.mark.parametrize("x", [-30.0, -4.0, -1.0, 0.0, 0.25, 1.0, 4.0, 30.0])
def test_silu_closed_forms(x):
    s = oracle.silu
    assert s(x) == pytest.approx(x / (1.0 + math.exp(-x)), rel=1e-14, abs=1e-300)
    assert s(x) - s(-x) == pytest.approx(x, rel=1e-12, abs=1e-15)
    assert oracle.silu(0.0) == 0.0


# ---------------------------------------------------------------- number formats

def test_bf16_matches_torch_rounding():
    x = np.concatenate([RNG.standard_normal(4000) * 10.0 ** RNG.integers(-30, 30, 4000),
                        [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 3e38]])
    x32 = x.astype(np.float32)
    ours = oracle.to_bf16_bits(x32.astype(np.float64))
    theirs = bf16_bits_from_f32(x32)
    assert np.array_equal(ours, theirs)


def test_bf16_ties_to_even():
    assert oracle.bf16_bits_to_f64(oracle.to_bf16_bits([1 + 2 ** -8]))[0] == 1.0
    assert oracle.bf16_bits_to_f64(oracle.to_bf16_bits([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6


def _golden_e4m3():
    rows = []
    with open(os.path.join(HERE, "golden", "e4m3_codes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            v = tok[0]
            if "2^" in v:
                coef, _, exp = v.partition("2^")
                coef = coef.rstrip("*")
                neg = coef.startswith("-")
                coef = coef.lstrip("-")
                val = (float(coef) if coef else 1.0) * 2.0 ** int(exp)
                val = -val if neg else val
            else:
                val = float(v)
            rows.append((val, int(tok[1], 16)))
    return rows


@pytest.mark.parametrize("value,code", _golden_e4m3())
def test_e4m3_golden_codes(value, code):
    assert int(oracle.to_e4m3([value])[0]) == code


def test_e4m3_matches_torch_in_range():
    x = np.concatenate([RNG.uniform(-448, 448, 3000), RNG.standard_normal(3000) * 0.01])
    ours = oracle.to_e4m3(x)
    theirs = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # x is exactly representable in fp32 except for rounding of the draw itself;
    # compare on the fp32 values both sides see.
    ours32 = oracle.to_e4m3(x.astype(np.float32).astype(np.float64))
    assert np.array_equal(ours32, theirs)
    assert ours.shape == theirs.shape


def test_e4m3_decode_encode_round_trip():
    for c in range(256):
        if c in (0x7F, 0xFF):
            assert math.isnan(oracle.e4m3_to_f64([c])[0])
            continue
        v = oracle.e4m3_to_f64([c])[0]
        assert int(oracle.to_e4m3([v])[0]) == c


# ---------------------------------------------------------------- epilogue ops

def brute_force(A, B, b_is_nk, program, alpha=1.0, bias=None, row_scale=None, aux=None,
                fp8_scale=1.0):
    """Pure-Python loops (independent of oracle.c) for tiny problems, with the
    tanh textbook form of GELU and a finite-difference-free GELU derivative
    written as d/dx of 0.5 x (1 + tanh(u))."""
    Af, Bf = f64(A), f64(B)
    M, K = Af.shape
    N = Bf.shape[0] if b_is_nk else Bf.shape[1]

    def acc(m, n):
        s = 0.0
        for k in range(K):
            s += Af[m, k] * (Bf[n, k] if b_is_nk else Bf[k, n])
        return s

    def gelu_grad(x):
        c = math.sqrt(2 / math.pi)
        u = c * (x + 0.044715 * x ** 3)
        t = math.tanh(u)
        return 0.5 * (1 + t) + 0.5 * x * (1 - t * t) * c * (1 + 3 * 0.044715 * x * x)

    def silu(x):
        return x / (1 + math.exp(-x))

    def ew(op, y, m, n):
        if op == "alpha":
            return alpha * y
        if op == "bias":
            return y + float(bias[n])
        if op == "row_scale":
            return y * float(row_scale[m])
        if op == "residual":
            return y + f64(aux)[m, n]
        if op == "gelu_tanh":
            return gelu_tanh_textbook(y)
        if op == "relu":
            return max(y, 0.0)
        if op == "silu":
            return silu(y)
        if op == "gelu_tanh_grad":
            return y * gelu_grad(f64(aux)[m, n])
        raise KeyError(op)

    pair = [i for i, op in enumerate(program) if op.startswith("pair_")]
    nout = N // 2 if pair else N
    out = {"y": np.zeros((M, nout)), "amax": 0.0, "col": np.zeros(nout), "row": np.zeros(M)}
    for m in range(M):
        for j in range(nout):
            if pair:
                ip = pair[0]
                g = int(program[ip].split(":")[1]) if ":" in program[ip] else 1
                cg = (j // g) * 2 * g + j % g
                cu = cg + g
                yg, yu = acc(m, cg), acc(m, cu)
                for op in program[:ip]:
                    yg, yu = ew(op, yg, m, cg), ew(op, yu, m, cu)
                y = (silu(yg) if program[ip].startswith("pair_swiglu") else yg) * yu
                rest = program[ip + 1:]
            else:
                y = acc(m, j)
                rest = program
            stored = None
            for op in rest:
                if op == "store_bf16":
                    stored = y
                elif op == "amax":
                    out["amax"] = max(out["amax"], abs(y))
                elif op == "col_sum":
                    out["col"][j] += y
                elif op.startswith("row_rms_unrounded"):
                    out["row"][m] += y * y  # the fp64 value itself
                elif op.startswith("row_rms"):
                    out["row"][m] += f64(bf16_bits_from_f32(np.array([y])))[0] ** 2
                elif op == "store_e4m3":
                    pass
                else:
                    y = ew(op, y, m, j)
            out["y"][m, j] = y if stored is None else stored
    return out


PROGRAMS = [
    (("alpha", "bias", "gelu_tanh", "amax", "store_bf16"), "kn"),
    (("pair_swiglu", "store_bf16"), "kn"),
    (("pair_swiglu:4", "store_bf16"), "kn"),
    (("alpha", "bias", "pair_swiglu", "store_bf16"), "kn"),
    (("alpha", "bias", "relu", "amax", "store_bf16", "store_e4m3"), "kn"),
    (("residual", "store_bf16", "row_rms:1e-6"), "kn"),
    (("residual", "store_bf16", "row_rms_unrounded:1e-6"), "kn"),
    (("alpha", "bias", "gelu_tanh", "store_bf16", "row_rms_unrounded:1e-3"), "nk"),
    (("gelu_tanh_grad", "store_bf16", "col_sum"), "nk"),
    (("row_scale", "silu", "store_bf16"), "nk"),
    (("row_scale", "pair_mul", "store_bf16"), "kn"),
    (("alpha", "pair_mul:2", "amax", "store_bf16"), "nk"),
]


@pytest.mark.parametrize("program,layout", PROGRAMS)
def test_oracle_matches_brute_force(program, layout):
    M, N, K = 5, 16, 9
    A = rand_bf16((M, K), 0.7)
    B = rand_bf16((K, N) if layout == "kn" else (N, K), 0.7)
    pair = any(op.startswith("pair") for op in program)
    nout = N // 2 if pair else N
    bias = None
    if "bias" in program:
        ip = next((i for i, op in enumerate(program) if op.startswith("pair")), None)
        bias_len = N if (ip is not None and program.index("bias") < ip) else nout
        bias = RNG.standard_normal(bias_len).astype(np.float32) * 0.1
    row_scale = RNG.uniform(0.5, 2.0, M).astype(np.float32)
    aux = rand_bf16((M, nout))
    uses_aux = "residual" in program or "gelu_tanh_grad" in program
    p = Problem(A, B, list(program), b_is_nk=(layout == "nk"), alpha=0.75, bias=bias,
                row_scale=row_scale, residual=aux if "residual" in program else None,
                preact=aux if "gelu_tanh_grad" in program else None, fp8_scale=112.0)
    got = p.rows()
    ref = brute_force(A, B, layout == "nk", list(program), alpha=0.75, bias=bias,
                      row_scale=row_scale, aux=aux if uses_aux else None)
    np.testing.assert_allclose(got["y"], ref["y"], rtol=1e-12, atol=1e-14)
    if "amax" in program:
        assert got["amax"] == pytest.approx(ref["amax"], rel=1e-12)
    if "col_sum" in program:
        cs = p.cols(list(range(nout)))
        np.testing.assert_allclose(cs["col_stat"], ref["col"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(cs["y"], got["y"], rtol=1e-15, atol=0)
    rms = [op for op in program if op.startswith("row_rms")]
    if rms:
        eps = float(rms[0].split(":")[1])
        want = 1.0 / np.sqrt(ref["row"] / nout + eps)
        np.testing.assert_allclose(got["row_stat"], want, rtol=1e-12)


def test_swapped_gate_up_is_caught():
    """Planted mistake: swapping gate and up (up * silu(gate) vs gate *
    silu(up)) must differ from the brute force."""
    A = rand_bf16((3, 6))
    B = rand_bf16((6, 8))
    good = brute_force(A, B, False, ["pair_swiglu", "store_bf16"])["y"]
    # Build the swapped version through the oracle by exchanging B's columns.
    Bs = B.copy()
    Bs[:, 0::2], Bs[:, 1::2] = B[:, 1::2], B[:, 0::2]
    swapped = Problem(A, Bs, ["pair_swiglu", "store_bf16"]).rows()["y"]
    assert not np.allclose(good, swapped, rtol=1e-6)


def test_swiglu_identity_pin():
    """A = I: out[m, j] = silu(B[m, 2j]) * B[m, 2j+1], values known exactly."""
    K = 8
    B = rand_bf16((K, 12))
    y = Problem(bf16_bits_from_f32(np.eye(K)), B, ["pair_swiglu", "store_bf16"]).rows()["y"]
    Bf = f64(B)
    want = Bf[:, 0::2] / (1 + np.exp(-Bf[:, 0::2])) * Bf[:, 1::2]
    np.testing.assert_allclose(y, want, rtol=1e-14)


def test_row_scale_rewrite_identity():
    """(X*S)@W == (X@W)*S for a row-broadcast S (powers of two keep X*S exact)."""
    M, K, N = 6, 10, 7
    X = rand_bf16((M, K))
    W = rand_bf16((K, N))
    S = (2.0 ** RNG.integers(-3, 4, M)).astype(np.float32)
    XS = bf16_bits_from_f32(f64(X) * S[:, None])
    lhs = Problem(XS, W, ["store_bf16"]).rows()["y"]
    rhs = Problem(X, W, ["row_scale", "store_bf16"], row_scale=S).rows()["y"]
    assert np.array_equal(lhs, rhs)


def test_row_rms_constant_rows_closed_form():
    M, K, N = 4, 8, 16
    A = np.zeros((M, K), np.uint16)
    B = rand_bf16((K, N))
    c = np.array([0.5, -2.0, 3.0, 0.0])
    res = bf16_bits_from_f32(np.repeat(c[:, None], N, 1))
    r = Problem(A, B, ["residual", "store_bf16", "row_rms:1e-6"], residual=res).rows()["row_stat"]
    np.testing.assert_allclose(r, 1 / np.sqrt(c * c + 1e-6), rtol=1e-15)


def _rms_rows(mode):
    """Rows whose epilogue value is 1 + 2^-10 in every column (B = 1, residual
    2^-10, A = I): exactly representable in fp64, but not in bf16, where it
    rounds to 1.  The two row-RMS modes must see different values."""
    M, N = 3, 24
    A = bf16_bits_from_f32(np.eye(M, 4))
    B = bf16_bits_from_f32(np.ones((4, N)))
    res = bf16_bits_from_f32(np.full((M, N), 2.0 ** -10))
    return Problem(A, B, ["residual", "store_bf16", mode + ":1e-6"], residual=res).rows()["row_stat"]


def test_row_rms_unrounded_closed_form():
    """row_rms_unrounded: S = 1/sqrt(mean(y^2) + eps) of the fp64 value
    ("Lean4-TileLang Tensor Program Superoptimizer", section 9, RMSNorm's S),
    here mean(y^2) = (1 + 2^-10)^2 in closed form; row_rms squares the bf16
    rounding of y, 1.0.  The pair differs by about 2^-10 relative, so squaring
    the rounded value in the unrounded mode (or the reverse) fails here."""
    y = 1.0 + 2.0 ** -10
    unrounded = _rms_rows("row_rms_unrounded")
    rounded = _rms_rows("row_rms")
    np.testing.assert_allclose(unrounded, 1.0 / math.sqrt(y * y + 1e-6), rtol=1e-15)
    np.testing.assert_allclose(rounded, 1.0 / math.sqrt(1.0 + 1e-6), rtol=1e-15)
    assert np.all(np.abs(unrounded / rounded - 1.0) > 5e-4)


def test_row_rms_unrounded_pure_python_mean():
    """A random row: the unrounded mode's statistic equals a pure-Python
    mean of the squared fp64 values the oracle reports, and differs from the
    mean of their bf16 roundings."""
    M, N, K = 4, 40, 12
    A = rand_bf16((M, K), 0.5)
    B = rand_bf16((K, N), 0.5)
    res = rand_bf16((M, N))
    p = Problem(A, B, ["residual", "store_bf16", "row_rms_unrounded:1e-6"], residual=res)
    out = p.rows()
    for m in range(M):
        ys = [float(v) for v in out["y"][m]]
        want = 1.0 / math.sqrt(sum(v * v for v in ys) / N + 1e-6)
        assert out["row_stat"][m] == pytest.approx(want, rel=1e-13)
        rounded = f64(bf16_bits_from_f32(np.array(ys)))
        wrong = 1.0 / math.sqrt(float(np.sum(rounded * rounded)) / N + 1e-6)
        assert abs(out["row_stat"][m] / wrong - 1.0) > 1e-6  # rounding changes this row


def test_amax_and_stores_consistent():
    A = rand_bf16((20, 32))
    B = rand_bf16((32, 24))
    bias = RNG.standard_normal(24).astype(np.float32)
    out = Problem(A, B, ["alpha", "bias", "relu", "amax", "store_bf16", "store_e4m3"],
                  alpha=0.5, bias=bias, fp8_scale=112.0).rows()
    assert out["amax"] == np.abs(out["y"]).max()
    assert np.all(out["y"] >= 0)
    assert np.array_equal(out["c_bf16"], oracle.to_bf16_bits(out["y"]))
    assert np.array_equal(out["c_e4m3"], oracle.to_e4m3(out["y"] * 112.0))
    # bf16(amax) equals the max of the stored bf16 values (rounding is monotone).
    assert oracle.to_bf16_bits([out["amax"]])[0] == out["c_bf16"].max()


def test_nan_input_row_is_nan_and_wins_amax():
    """A NaN operand element makes its row's outputs NaN (bf16 NaN, e4m3 NaN
    code) and the AMAX NaN; the other rows are untouched."""
    A = rand_bf16((6, 8))
    B = rand_bf16((8, 16))
    A[2, 5] = 0x7FC0  # bf16 quiet NaN
    out = Problem(A, B, ["gelu_tanh", "amax", "store_bf16", "store_e4m3"], fp8_scale=8.0).rows()
    assert np.all(np.isnan(out["y"][2]))
    assert np.all((out["c_bf16"][2] & 0x7FFF) > 0x7F80)  # NaN bit patterns
    assert np.all((out["c_e4m3"][2] & 0x7F) == 0x7F)
    assert math.isnan(out["amax"])
    clean = Problem(np.delete(A, 2, 0), B, ["gelu_tanh", "amax", "store_bf16"]).rows()
    np.testing.assert_array_equal(np.delete(out["y"], 2, 0), clean["y"])


def test_cols_match_rows():
    A = rand_bf16((9, 16))
    W = rand_bf16((12, 16))
    pre = rand_bf16((9, 12))
    p = Problem(A, W, ["gelu_tanh_grad", "store_bf16", "col_sum"], b_is_nk=True, preact=pre)
    rows = p.rows()["y"]
    cols = p.cols([0, 3, 11])
    np.testing.assert_array_equal(cols["y"], rows[:, [0, 3, 11]])
    np.testing.assert_allclose(cols["col_stat"], rows[:, [0, 3, 11]].sum(0), rtol=1e-13)


def test_bad_program_rejected():
    A = rand_bf16((2, 2))
    with pytest.raises(ValueError):
        Problem(A, A, ["no_such_op"]).rows()


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("pair", ["pair_swiglu:128", "pair_mul:128"])
def test_two_weight_pairs_match_numpy(layout, pair):
    """With a second weight operand and pair group 128, out = f(A@W_gate) *
    (A@W_up) (Superoptimizer, section 7: gate = X @ W_gate, up = X @ W_up)."""
    M, K, H = 5, 24, 384
    A = rand_bf16((M, K))
    Wg = rand_bf16((K, H) if layout == "kn" else (H, K))
    Wu = rand_bf16((K, H) if layout == "kn" else (H, K))
    p = Problem(A, Wg, [pair, "store_bf16"], b_is_nk=(layout == "nk"), B2=Wu)
    assert p.out_cols() == H
    y = p.rows()["y"]
    G = f64(A) @ (f64(Wg) if layout == "kn" else f64(Wg).T)
    U = f64(A) @ (f64(Wu) if layout == "kn" else f64(Wu).T)
    f = G / (1 + np.exp(-G)) if pair.startswith("pair_swiglu") else G
    np.testing.assert_allclose(y, f * U, rtol=1e-12, atol=1e-14)
    cols = p.cols([0, 127, 128, 383])
    np.testing.assert_allclose(cols["y"], y[:, [0, 127, 128, 383]], rtol=1e-15)


# ---------------------------------------------------------------- FP8 operands

def _torch_decode(codes, dtype):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(dtype)
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("name,dtype", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_decode_matches_torch_for_every_code(name, dtype):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes) if name == "e4m3" else oracle.e5m2_to_f64(codes)
    theirs = _torch_decode(codes, dtype)
    assert np.array_equal(np.isnan(ours), np.isnan(theirs))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], theirs[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(theirs[ok]))


def test_e5m2_closed_forms():
    # 1.0, largest finite (1.75 * 2^15), smallest subnormal (2^-16), smallest
    # normal (2^-14), -2, +inf, a NaN.
    vals = oracle.e5m2_to_f64(np.array([0x3C, 0x7B, 0x01, 0x04, 0xC0, 0x7C, 0x7D], np.uint8))
    assert list(vals[:6]) == [1.0, 57344.0, 2.0 ** -16, 2.0 ** -14, -2.0, math.inf]
    assert math.isnan(vals[6])


def _rand_fp8(shape, dtype, scale):
    t = torch.from_numpy((RNG.standard_normal(shape) * scale).astype(np.float32)).to(dtype)
    return t.view(torch.uint8).numpy()


@pytest.mark.parametrize("a_t,b_t", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_fp8_gemm_matches_numpy_einsum(a_t, b_t, layout):
    """Codes decoded by torch, multiplied by numpy in fp64, then scaled by
    both dequantisation factors (distinct, so a dropped one shows)."""
    dt = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
    M, N, K = 13, 21, 48
    A = _rand_fp8((M, K), dt[a_t], 30.0)
    B = _rand_fp8((K, N) if layout == "kn" else (N, K), dt[b_t], 30.0)
    sa, sb = 1.0 / 30.0, 1.0 / 112.0
    y = Problem(A, B, ["store_bf16"], b_is_nk=(layout == "nk"), a_type=a_t, b_type=b_t,
                a_scale_inv=sa, b_scale_inv=sb).rows()["y"]
    Ad = _torch_decode(A, dt[a_t])
    Bd = _torch_decode(B, dt[b_t])
    ref = np.einsum("mk,kn->mn", Ad, Bd if layout == "kn" else Bd.T) * sa * sb
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)


def test_fp8_scale_applies_before_the_program():
    """relu(alpha * acc + bias) with the dequantisation inside acc: a bias
    added before the scaling would give a different result."""
    A = np.full((2, 16), 0x38, np.uint8)            # e4m3 1.0
    B = np.full((16, 3), 0x40, np.uint8)            # e4m3 2.0
    bias = np.array([-1.0, 0.0, 1.0], np.float32)
    r = Problem(A, B, ["alpha", "bias", "relu", "store_bf16"], alpha=0.5, bias=bias, a_type="e4m3",
                b_type="e4m3", a_scale_inv=0.25, b_scale_inv=0.5).rows()
    # acc = 0.25 * 0.5 * 16 * 2 = 4; y = relu(0.5 * 4 + bias)
    assert np.array_equal(r["y"], np.array([[1.0, 2.0, 3.0]] * 2))


def test_fp8_operand_type_is_enforced():
    with pytest.raises(TypeError):
        Problem(rand_bf16((2, 16)), np.zeros((16, 2), np.uint8), [], a_type="e4m3", b_type="e4m3").rows()


# ---------------------------------------------------------------- dSwiGLU

@pytest.mark.parametrize("x", [-20.0, -3.0, -1.0, -0.2, 0.0, 0.3, 1.0, 2.5, 20.0])
def test_silu_grad_closed_forms(x):
    d = oracle.silu_grad(x)
    assert oracle.silu_grad(0.0) == 0.5
    assert abs(d + oracle.silu_grad(-x) - 1.0) < 1e-14       # silu(x) - silu(-x) = x
    h = 1e-5
    fd = (oracle.silu(x + h) - oracle.silu(x - h)) / (2 * h)  # central difference
    assert abs(d - fd) < 1e-8


def _dswiglu_case(M, N, K, g, seed):
    rng = np.random.default_rng(seed)
    A = bf16_bits_from_f32(rng.standard_normal((M, K)) * 0.5)
    B = bf16_bits_from_f32(rng.standard_normal((K, N)) * 0.5)
    pre = bf16_bits_from_f32(rng.standard_normal((M, 2 * N)) * 1.5)
    return A, B, pre


@pytest.mark.parametrize("g", [1, 2, 4, 16])
def test_dswiglu_matches_autograd(g):
    """The backward of h = silu(gate) * up by torch autograd (fp64), with dh
    the GEMM result: both gradients land on the forward's interleaved gate /
    up positions."""
    M, N, K = 5, 32, 12
    A, B, pre = _dswiglu_case(M, N, K, g, 40 + g)
    y = Problem(A, B, ["dswiglu:%d" % g, "store_bf16"], preact=pre).rows()["y"]
    P = torch.from_numpy(f64(pre))
    cols = np.arange(N)
    cg = (cols // g) * 2 * g + cols % g
    gate = P[:, cg].clone().requires_grad_(True)
    up = P[:, cg + g].clone().requires_grad_(True)
    dh = torch.from_numpy(f64(A) @ f64(B))
    (torch.nn.functional.silu(gate) * up).backward(dh)
    ref = np.zeros((M, 2 * N))
    ref[:, cg] = gate.grad.numpy()
    ref[:, cg + g] = up.grad.numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_dswiglu_brute_force_with_pre_and_post_ops():
    """Pure-Python loops: alpha and a row scale on dh (accumulator columns),
    then bias on the 2N output columns, AMAX, bf16 store and column sums."""
    M, N, K, g = 3, 8, 6, 2
    A, B, pre = _dswiglu_case(M, N, K, g, 50)
    rs = np.array([0.5, 2.0, -1.0], np.float32)
    bias = np.linspace(-1, 1, 2 * N).astype(np.float32)
    prog = ["alpha", "row_scale", "dswiglu:2", "bias", "amax", "store_bf16", "col_sum"]
    p = Problem(A, B, prog, alpha=0.75, row_scale=rs, bias=bias, preact=pre)
    r = p.rows()
    c = p.cols(list(range(2 * N)))
    Af, Bf, Pf = f64(A), f64(B), f64(pre)
    want = np.zeros((M, 2 * N))
    for m in range(M):
        for o in range(2 * N):
            j = (o // (2 * g)) * g + o % g
            dh = sum(Af[m, k] * Bf[k, j] for k in range(K)) * 0.75 * float(rs[m])
            base = (o // (2 * g)) * 2 * g + o % g
            gt, up = Pf[m, base], Pf[m, base + g]
            sg = 1.0 / (1.0 + math.exp(-gt))
            if o % (2 * g) < g:
                v = dh * up * (sg + gt * sg * (1 - sg))
            else:
                v = dh * gt * sg
            want[m, o] = v + float(bias[o])
    np.testing.assert_allclose(r["y"], want, rtol=1e-12, atol=1e-13)
    assert abs(r["amax"] - np.abs(want).max()) < 1e-12
    np.testing.assert_allclose(c["col_stat"], want.sum(0), rtol=1e-12, atol=1e-12)


def test_dswiglu_swapped_gate_up_is_caught():
    """Swapping the gate and up inputs changes the result, so the autograd
    pin above would catch it."""
    M, N, K = 2, 4, 4
    A, B, pre = _dswiglu_case(M, N, K, 1, 60)
    swapped = pre.copy()
    swapped[:, 0::2], swapped[:, 1::2] = pre[:, 1::2], pre[:, 0::2]
    y1 = Problem(A, B, ["dswiglu", "store_bf16"], preact=pre).rows()["y"]
    y2 = Problem(A, B, ["dswiglu", "store_bf16"], preact=swapped).rows()["y"]
    assert np.abs(y1 - y2).max() > 1e-3


# ---------------------------------------------------------------- RMSNorm backward

def _rmsnorm_case(M, D, seed):
    rng = np.random.default_rng(seed)
    x = bf16_bits_from_f32(rng.standard_normal((M, D)) * 2.0 + 0.3)
    dy = bf16_bits_from_f32(rng.standard_normal((M, D)))
    w = (rng.standard_normal(D) * 0.5 + 1.0).astype(np.float32)
    return x, dy, w


@pytest.mark.parametrize("M,D", [(3, 8), (5, 48)])
def test_rmsnorm_backward_matches_autograd(M, D):
    """dy arrives as a GEMM result (dy @ I); the epilogue's col_scale (w) and
    row_dot (sum w dy x) feed the finishing step; dx and dw equal torch
    autograd of y = x * (mean x^2 + eps)^(-1/2) * w in fp64."""
    eps = 1e-6
    x, dy, w = _rmsnorm_case(M, D, 90 + D)
    xf = f64(x)
    S = (1.0 / np.sqrt((xf * xf).mean(1) + eps)).astype(np.float32)
    eye = bf16_bits_from_f32(np.eye(D))
    r = Problem(dy, eye, ["store_bf16", "col_scale", "row_dot"], col_scale=w, residual=x).rows()["row_stat"]
    dx, dw = oracle.rmsnorm_backward(dy, x, S, r, w=w)
    xt = torch.from_numpy(xf).requires_grad_(True)
    wt = torch.from_numpy(w.astype(np.float64)).requires_grad_(True)
    St = torch.from_numpy(S.astype(np.float64))  # the forward's S as stored (fp32)
    # S as a function of x for autograd, pinned to the stored fp32 value
    Sx = torch.rsqrt((xt * xt).mean(1) + eps)
    y = xt * (Sx + (St - Sx).detach())[:, None] * wt
    y.backward(torch.from_numpy(f64(dy)))
    # S enters the finishing step as the stored fp32 value (2^-24 relative
    # from the fp64 one autograd differentiates, cubed in the second term).
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-6, atol=1e-6 * np.abs(dx).max())
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-6, atol=1e-6 * np.abs(dw).max())


def test_row_dot_and_col_scale_brute_force():
    M, N, K = 3, 6, 5
    rng = np.random.default_rng(95)
    A = bf16_bits_from_f32(rng.standard_normal((M, K)))
    B = bf16_bits_from_f32(rng.standard_normal((K, N)))
    x = bf16_bits_from_f32(rng.standard_normal((M, N)))
    cs = rng.standard_normal(N).astype(np.float32)
    r = Problem(A, B, ["alpha", "col_scale", "store_bf16", "row_dot"], alpha=0.5, col_scale=cs,
                residual=x).rows()
    Af, Bf, xf = f64(A), f64(B), f64(x)
    want_y = np.zeros((M, N))
    want_r = np.zeros(M)
    for m in range(M):
        for n in range(N):
            v = sum(Af[m, k] * Bf[k, n] for k in range(K)) * 0.5 * float(cs[n])
            want_y[m, n] = v
            want_r[m] += v * xf[m, n]
    np.testing.assert_allclose(r["y"], want_y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["row_stat"], want_r, rtol=1e-12, atol=1e-12)


def test_rmsnorm_backward_add_term_and_unit_weight():
    M, D = 4, 16
    x, dy, _ = _rmsnorm_case(M, D, 97)
    add = bf16_bits_from_f32(np.arange(M * D, dtype=np.float64).reshape(M, D) / 64)
    S = np.full(M, 0.5, np.float32)
    r = np.linspace(-1, 1, M)
    dx0, dw0 = oracle.rmsnorm_backward(dy, x, S, r)          # w = 1
    dx1, _ = oracle.rmsnorm_backward(dy, x, S, r, add=add)
    np.testing.assert_allclose(dx1 - dx0, f64(add), rtol=0, atol=1e-15)
    want = 0.5 * f64(dy) - f64(x) * (0.125 * r / D)[:, None]
    np.testing.assert_allclose(dx0, want, rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(dw0, (f64(dy) * f64(x) * 0.5).sum(0), rtol=1e-14)
