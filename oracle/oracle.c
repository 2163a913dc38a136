/*
 * oracle.c -- plain, slow, fp64 CPU reference of the fused GEMM + epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no source, header, table or constant with the CUDA path under
 * gemm_epilogue_transformer_smem_gb300/ and the product never calls it.
 *
 * What it computes (one definition, no blocking, no fusion, no reordering):
 *
 *   acc[m,n] = sa * sb * sum_k A[m,k] * B[k,n]          (fp64, exact widening
 *                                                         of the bf16 / fp8
 *                                                         inputs; sa, sb the
 *                                                         operands' dequant
 *                                                         factors, 1 for bf16)
 *   then the epilogue program, op by op, in the order given, per element.
 *
 * Sources, cited by page title and section:
 *  - GEMM O = X @ W: "Lean4-TileLang Tensor Program Superoptimizer"
 *    (itsolotime.com), section 8 "Matmul".
 *  - bias + GELU finished on the accumulator before the store:
 *    "Toi uu hoa GPU Kernel voi TileLang: Tu GEMM den FlashAttention"
 *    (aihot.vn), the fused GEMM epilogue paragraph.
 *  - alpha (host scalar) * acc + bias -> activation -> AMAX of the result, for
 *    the next FP8 quantisation: "Huong dan su dung NVIDIA cuDNN Graph API"
 *    (aihot.vn), the batched matmul epilogue paragraph.
 *  - SwiGLU out = up * silu(gate), silu(x) = x * sigmoid(x): Superoptimizer,
 *    section 7 "SwiGLU"; the RMSNorm-MLP's plain out = up * gate:
 *    Superoptimizer, section 10 "RMSNorm-MLP".
 *  - RMSNorm scale S = 1 / sqrt(mean(x^2) + eps) and the row-broadcast rewrite
 *    (X*S)@W = (X@W)*S: Superoptimizer, sections 3 and 9 "RMSNorm".
 *  - scaling, reductions, pairwise transforms and accumulation applied to the
 *    output tile, forward and backward: "CODA: ... GEMM-Epilogue"
 *    (lehuy.net), "How CODA works".
 *
 * Readings where the pages are silent:
 *  - GELU is the tanh approximation 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715
 *    x^3))), evaluated as x * sigmoid(2u); its derivative is
 *    s + 2 x s (1 - s) sqrt(2/pi) (1 + 3*0.044715 x^2), s = sigmoid(2u).
 *  - pair_swiglu(g) / pair_mul(g): output column j takes gate from
 *    accumulator column (j/g)*2g + j%g and up from (j/g)*2g + g + j%g; g = 1
 *    is even/odd.
 *  - col_scale: y * col_scale[n] (a per-column scaling, e.g. an RMSNorm
 *    weight); row_dot: row_stat[m] = sum_n y * residual[m, n], the row
 *    reduction of the RMSNorm backward (the CODA page's reductions on the
 *    output tile); oracle_rmsnorm_backward finishes dx and dw from it.
 *  - dswiglu(g), the backward of pair_swiglu(g) (CODA's backward epilogues:
 *    a pairwise transform producing both gradients): the accumulator holds
 *    dh for h = silu(gate) * up; the forward pre-activations (gate, up) are
 *    read from `preact` at the same interleaved positions (2N columns), and
 *    output columns gate(j), up(j) receive dh * up * silu'(gate) and
 *    dh * silu(gate), silu'(x) = sigmoid(x) (1 + x (1 - sigmoid(x))).
 *  - e4m3 is OCP FP8 E4M3FN (bias 7, max 448, no infinities); quantisation is
 *    round-to-nearest-even of value*scale, saturated to +-448, NaN kept.
 *  - FP8 operands (the FP8 training loop of the cuDNN Graph API tutorial's
 *    matmul epilogue paragraph: an AMAX-derived scale quantises the next
 *    GEMM's input): e4m3 or e5m2 codes (OCP E5M2: bias 15, infinities and
 *    NaNs at exponent 31) widened exactly; each operand's per-tensor
 *    dequantisation factor (the reciprocal of its quantisation scale)
 *    multiplies the accumulator.
 *  - row_rms averages the squares of the bf16-rounded values (what the next
 *    RMSNorm reads); row_rms_unrounded squares the fp64 values.  col_sum and
 *    amax observe the unrounded value.
 *
 * Parity pins: tests/test_oracle_pins.py checks this file against numpy,
 * closed forms, identity/permutation inputs, hand-derived e4m3 codes and a
 * pure-Python brute force.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

/* ------------------------------------------------------------------ */
/* number formats                                                      */
/* ------------------------------------------------------------------ */

double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* bf16 = 1 sign, 8 exponent (bias 127), 7 fraction bits.  Round to nearest,
 * ties to even, directly from the fp64 value (no intermediate fp32). */
uint16_t oracle_double_to_bf16(double x)
{
    if (isnan(x)) return 0x7FC0;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs(x);
    uint16_t sign = (uint16_t)(neg << 15);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    frexp(a, &e);           /* a = f * 2^e, f in [0.5, 1) -> floor(log2 a) = e-1 */
    int ex = e - 1;
    if (ex < -126) ex = -126;           /* subnormal spacing below 2^-126 */
    double ulp = ldexp(1.0, ex - 7);
    double q = nearbyint(a / ulp) * ulp; /* default rounding mode: ties to even */
    double maxfin = ldexp(255.0, 127 - 7); /* (2 - 2^-7) * 2^127 */
    if (q > maxfin) return (uint16_t)(sign | 0x7F80);
    float f = (float)q;                  /* exact: q has <= 8 significant bits */
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(sign | (uint16_t)((w >> 16) & 0x7FFF));
}

/* e4m3 (OCP E4M3FN): 1 sign, 4 exponent (bias 7), 3 fraction bits.  Normal
 * values (1 + f/8) 2^(e-7) for e = 1..15 except e=15,f=7 (NaN); subnormals
 * f/8 * 2^-6.  Largest finite 448.  Round to nearest even, then saturate. */
uint8_t oracle_double_to_e4m3(double x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a == 0.0) return sign;
    double q;
    if (isinf(a)) {
        q = 448.0;
    } else {
        int e;
        frexp(a, &e);
        int ex = e - 1;
        if (ex < -6) ex = -6;             /* subnormal spacing 2^-9 */
        double ulp = ldexp(1.0, ex - 3);
        q = nearbyint(a / ulp) * ulp;
        if (q > 448.0) q = 448.0;         /* satfinite */
    }
    if (q == 0.0) return sign;
    int e;
    frexp(q, &e);
    int ex = e - 1;
    uint8_t code;
    if (ex < -6) {
        code = (uint8_t)nearbyint(q / ldexp(1.0, -9));           /* 1..7 */
    } else {
        int frac = (int)nearbyint((q / ldexp(1.0, ex) - 1.0) * 8.0); /* 0..7 */
        code = (uint8_t)(((ex + 7) << 3) | frac);
    }
    return (uint8_t)(sign | code);
}

double oracle_e4m3_to_double(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, f = c & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) v = ldexp((double)f / 8.0, -6);
    else v = ldexp(1.0 + (double)f / 8.0, e - 7);
    return s ? -v : v;
}

/* e5m2 (OCP E5M2): 1 sign, 5 exponent (bias 15), 2 fraction bits.  Normal
 * values (1 + f/4) 2^(e-15) for e = 1..30; exponent 31 is infinity (f = 0)
 * or NaN; subnormals f/4 * 2^-14.  Largest finite 57344. */
double oracle_e5m2_to_double(uint8_t c)
{
    int s = c >> 7, e = (c >> 2) & 0x1F, f = c & 3;
    double v;
    if (e == 31) {
        if (f) return NAN;
        v = INFINITY;
    } else if (e == 0) {
        v = ldexp((double)f / 4.0, -14);
    } else {
        v = ldexp(1.0 + (double)f / 4.0, e - 15);
    }
    return s ? -v : v;
}

/* ------------------------------------------------------------------ */
/* activations (fp64)                                                  */
/* ------------------------------------------------------------------ */

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

static const double GELU_C = 0.044715;

static double gelu_u(double x)
{
    return sqrt(2.0 / M_PI) * (x + GELU_C * x * x * x);
}

double oracle_gelu_tanh(double x) { return x * sigmoid(2.0 * gelu_u(x)); }

double oracle_gelu_tanh_grad(double x)
{
    double s = sigmoid(2.0 * gelu_u(x));
    double du = sqrt(2.0 / M_PI) * (1.0 + 3.0 * GELU_C * x * x);
    return s + 2.0 * x * s * (1.0 - s) * du;
}

double oracle_silu(double x) { return x * sigmoid(x); }

/* d/dx [x sigmoid(x)] = sigmoid(x) (1 + x (1 - sigmoid(x))). */
double oracle_silu_grad(double x)
{
    double s = sigmoid(x);
    return s * (1.0 + x * (1.0 - s));
}

/* ------------------------------------------------------------------ */
/* program parsing                                                     */
/* ------------------------------------------------------------------ */

enum {
    O_ALPHA, O_BIAS, O_ROW_SCALE, O_RESIDUAL, O_GELU, O_RELU, O_SILU, O_PAIR,
    O_PAIR_MUL, O_GELU_GRAD, O_AMAX, O_STORE_BF16, O_STORE_E4M3, O_ROW_RMS, O_COL_SUM,
    O_DSWIGLU, O_COL_SCALE, O_ROW_DOT
};

typedef struct { int code; double f; int i; } oop;

#define ORACLE_MAX_OPS 32

/* "name" or "name:number" separated by commas, e.g.
 * "alpha,bias,gelu_tanh,amax,store_bf16" or "residual,store_bf16,row_rms:1e-6" */
static int parse_program(const char *s, oop *ops, int *n_out)
{
    /* mode: row_rms squares the bf16-rounded value, row_rms_unrounded the
     * fp64 value. */
    static const struct { const char *name; int code; int mode; } names[] = {
        {"alpha", O_ALPHA, 0}, {"bias", O_BIAS, 0}, {"row_scale", O_ROW_SCALE, 0},
        {"residual", O_RESIDUAL, 0}, {"gelu_tanh", O_GELU, 0}, {"relu", O_RELU, 0},
        {"silu", O_SILU, 0}, {"pair_swiglu", O_PAIR, 0}, {"pair_mul", O_PAIR_MUL, 0},
        {"gelu_tanh_grad", O_GELU_GRAD, 0}, {"amax", O_AMAX, 0},
        {"store_bf16", O_STORE_BF16, 0}, {"store_e4m3", O_STORE_E4M3, 0},
        {"row_rms", O_ROW_RMS, 0}, {"row_rms_unrounded", O_ROW_RMS, 1},
        {"col_sum", O_COL_SUM, 0}, {"dswiglu", O_DSWIGLU, 0},
        {"col_scale", O_COL_SCALE, 0}, {"row_dot", O_ROW_DOT, 0},
    };
    int n = 0;
    const char *p = s ? s : "";
    while (*p) {
        char tok[64];
        size_t len = strcspn(p, ",");
        if (len == 0 || len >= sizeof tok) return -1;
        memcpy(tok, p, len);
        tok[len] = 0;
        p += len;
        if (*p == ',') ++p;
        char *colon = strchr(tok, ':');
        double f = 0.0;
        int has_arg = 0;
        if (colon) { *colon = 0; f = strtod(colon + 1, NULL); has_arg = 1; }
        int code = -1, mode = 0;
        for (size_t i = 0; i < sizeof names / sizeof names[0]; ++i)
            if (strcmp(tok, names[i].name) == 0) { code = names[i].code; mode = names[i].mode; }
        if (code < 0 || n >= ORACLE_MAX_OPS) return -1;
        ops[n].code = code;
        ops[n].f = f;
        ops[n].i = code == O_ROW_RMS ? mode : (int)f;
        /* defaults */
        if ((code == O_PAIR || code == O_PAIR_MUL || code == O_DSWIGLU) && !has_arg)
            ops[n].i = 1; /* group g */
        if ((code == O_PAIR || code == O_PAIR_MUL || code == O_DSWIGLU) && ops[n].i < 1) return -1;
        if (code == O_ROW_RMS && !has_arg) ops[n].f = 1e-6;     /* eps */
        ++n;
    }
    *n_out = n;
    return 0;
}

/* ------------------------------------------------------------------ */
/* the GEMM                                                            */
/* ------------------------------------------------------------------ */

/* Element i of an operand of the given type, widened exactly. */
static double elem_at(const void *base, int type, int64_t i)
{
    switch (type) {
    case ORACLE_E4M3: return oracle_e4m3_to_double(((const uint8_t *)base)[i]);
    case ORACLE_E5M2: return oracle_e5m2_to_double(((const uint8_t *)base)[i]);
    default: return oracle_bf16_to_double(((const uint16_t *)base)[i]);
    }
}

static double a_at(const oracle_problem *p, int64_t m, int64_t k)
{
    return elem_at(p->A, p->a_type, m * p->lda + k);
}

/* Accumulator column n.  With a second weight operand B2 the columns
 * alternate in blocks of 128: block 2i is B's columns [128i, 128i+128),
 * block 2i+1 is B2's same columns. */
static double b_at(const oracle_problem *p, int64_t k, int64_t n)
{
    const void *src = p->B;
    if (p->B2) {
        if ((n / 128) % 2) src = p->B2;
        n = (n / 256) * 128 + n % 128;
    }
    return p->b_is_nk ? elem_at(src, p->b_type, n * p->ldb + k)
                      : elem_at(src, p->b_type, k * p->ldb + n);
}

/* One whole accumulator row, i-k-j order for the K x N layout. */
static void acc_row(const oracle_problem *p, int64_t m, double *acc)
{
    for (int64_t n = 0; n < p->N; ++n) acc[n] = 0.0;
    if (!p->b_is_nk && !p->B2) {
        for (int64_t k = 0; k < p->K; ++k) {
            double a = a_at(p, m, k);
            for (int64_t n = 0; n < p->N; ++n)
                acc[n] += a * elem_at(p->B, p->b_type, k * p->ldb + n);
        }
    } else {
        for (int64_t n = 0; n < p->N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < p->K; ++k) s += a_at(p, m, k) * b_at(p, k, n);
            acc[n] = s;
        }
    }
    for (int64_t n = 0; n < p->N; ++n) acc[n] *= p->a_scale_inv * p->b_scale_inv;
}

/* One accumulator element. */
static double acc_elem(const oracle_problem *p, int64_t m, int64_t n)
{
    double s = 0.0;
    for (int64_t k = 0; k < p->K; ++k) s += a_at(p, m, k) * b_at(p, k, n);
    return s * p->a_scale_inv * p->b_scale_inv;
}

/* ------------------------------------------------------------------ */
/* the epilogue, one output element at a time                          */
/* ------------------------------------------------------------------ */

typedef struct {
    double stored;   /* value at store_bf16 (or the final value) */
    int has_store;
    uint16_t bf16;
    uint8_t e4m3;
    double amax;     /* |value| at amax, or 0 */
    double row_sq;   /* square used by row_rms */
    double row_dot;  /* value * residual at row_dot */
    double col_v;    /* value at col_sum */
} elem_out;

static int find_pair(const oop *ops, int n)
{
    for (int i = 0; i < n; ++i)
        if (ops[i].code == O_PAIR || ops[i].code == O_PAIR_MUL) return i;
    return -1;
}

/* Element-wise op on value y at (m, col).  Returns 0, or -1 for an output op
 * (handled by the caller). */
static double apply_elementwise(const oracle_problem *p, const oop *op, double y,
                                int64_t m, int64_t col)
{
    switch (op->code) {
    case O_ALPHA: return p->alpha * y;
    case O_BIAS: return y + (double)p->bias[col];
    case O_COL_SCALE: return y * (double)p->col_scale[col];
    case O_ROW_SCALE: return y * (double)p->row_scale[m];
    case O_RESIDUAL: return y + oracle_bf16_to_double(p->residual[m * p->ld_aux + col]);
    case O_GELU: return oracle_gelu_tanh(y);
    case O_RELU: return y > 0.0 ? y : 0.0;
    case O_SILU: return oracle_silu(y);
    case O_GELU_GRAD:
        return y * oracle_gelu_tanh_grad(oracle_bf16_to_double(p->preact[m * p->ld_aux + col]));
    default: return y;
    }
}

static int find_expand(const oop *ops, int n)
{
    for (int i = 0; i < n; ++i)
        if (ops[i].code == O_DSWIGLU) return i;
    return -1;
}

/* dswiglu(g): output column o of the 2N columns is the gate or the up
 * position of one forward pair; it takes accumulator column
 * j = (o / 2g) g + o % g (the gradient of silu(gate) * up at that pair). */
static int64_t expand_acc_col(int64_t o, int64_t g)
{
    return (o / (2 * g)) * g + o % g;
}

static void run_elem(const oracle_problem *p, const oop *ops, int nops, int64_t m,
                     int64_t j, double acc_a, double acc_b, elem_out *o)
{
    int ip = find_pair(ops, nops);
    int ie = find_expand(ops, nops);
    int first_post = 0;
    double y;
    memset(o, 0, sizeof *o);
    if (ie >= 0) {
        /* j is the output column; acc_a the accumulator at expand_acc_col(j).
         * Forward: h = silu(gate) * up.  Backward with dh = y:
         *   d gate = dh * up * silu'(gate),  d up = dh * silu(gate). */
        int64_t g = ops[ie].i;
        int64_t jacc = expand_acc_col(j, g);
        int64_t cg = (j / (2 * g)) * 2 * g + j % g;  /* gate position of the pair */
        int is_gate = (j % (2 * g)) < g;
        y = acc_a;
        for (int i = 0; i < ie; ++i) y = apply_elementwise(p, &ops[i], y, m, jacc);
        double gate = oracle_bf16_to_double(p->preact[m * p->ld_aux + cg]);
        double up = oracle_bf16_to_double(p->preact[m * p->ld_aux + cg + g]);
        y = is_gate ? y * up * oracle_silu_grad(gate) : y * oracle_silu(gate);
        first_post = ie + 1;
    } else if (ip >= 0) {
        int64_t g = ops[ip].i;
        int64_t cg = (j / g) * 2 * g + j % g, cu = cg + g;
        double yg = acc_a, yu = acc_b;
        for (int i = 0; i < ip; ++i) {
            yg = apply_elementwise(p, &ops[i], yg, m, cg);
            yu = apply_elementwise(p, &ops[i], yu, m, cu);
        }
        y = ops[ip].code == O_PAIR ? oracle_silu(yg) * yu : yg * yu;
        first_post = ip + 1;
    } else {
        y = acc_a;
    }
    for (int i = first_post; i < nops; ++i) {
        const oop *op = &ops[i];
        switch (op->code) {
        case O_STORE_BF16:
            o->stored = y;
            o->has_store = 1;
            o->bf16 = oracle_double_to_bf16(y);
            break;
        case O_STORE_E4M3: o->e4m3 = oracle_double_to_e4m3(y * p->fp8_scale); break;
        case O_AMAX: o->amax = fabs(y); break;
        case O_ROW_RMS: {
            double v = op->i == 1 ? y : oracle_bf16_to_double(oracle_double_to_bf16(y));
            o->row_sq = v * v;
            break;
        }
        case O_COL_SUM: o->col_v = y; break;
        case O_ROW_DOT: o->row_dot = y * oracle_bf16_to_double(p->residual[m * p->ld_aux + j]); break;
        default: y = apply_elementwise(p, op, y, m, j); break;
        }
    }
    if (!o->has_store) o->stored = y;
}

static int64_t out_cols(const oracle_problem *p, const oop *ops, int n)
{
    if (find_expand(ops, n) >= 0) return 2 * p->N;
    return find_pair(ops, n) >= 0 ? p->N / 2 : p->N;
}

static double row_rms_eps(const oop *ops, int n)
{
    for (int i = 0; i < n; ++i)
        if (ops[i].code == O_ROW_RMS) return ops[i].f;
    return 0.0;
}

int oracle_out_cols(const oracle_problem *p)
{
    oop ops[ORACLE_MAX_OPS];
    int n;
    if (parse_program(p->program, ops, &n)) return -1;
    return (int)out_cols(p, ops, n);
}

int oracle_rows(const oracle_problem *p, const int64_t *rows, int64_t nrows,
                double *y, uint16_t *c_bf16, uint8_t *c_e4m3, double *row_stat,
                double *amax_rows)
{
    oop ops[ORACLE_MAX_OPS];
    int nops;
    if (parse_program(p->program, ops, &nops)) return -1;
    int ip = find_pair(ops, nops);
    int ie = find_expand(ops, nops);
    int64_t nout = out_cols(p, ops, nops);
    double eps = row_rms_eps(ops, nops);
    int has_row_dot = 0;
    for (int i = 0; i < nops; ++i)
        if (ops[i].code == O_ROW_DOT) has_row_dot = 1;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows ? rows[r] : r;
        if (m < 0 || m >= p->M) { bad = 1; continue; }
        double *acc = (double *)malloc(sizeof(double) * (size_t)(p->N > 0 ? p->N : 1));
        if (!acc) { bad = 1; continue; }
        acc_row(p, m, acc);
        double ss = 0.0, am = 0.0, rd = 0.0;
        for (int64_t j = 0; j < nout; ++j) {
            elem_out o;
            if (ie >= 0) {
                run_elem(p, ops, nops, m, j, acc[expand_acc_col(j, ops[ie].i)], 0.0, &o);
            } else if (ip >= 0) {
                int64_t g = ops[ip].i;
                int64_t cg = (j / g) * 2 * g + j % g;
                run_elem(p, ops, nops, m, j, acc[cg], acc[cg + g], &o);
            } else {
                run_elem(p, ops, nops, m, j, acc[j], 0.0, &o);
            }
            if (y) y[r * nout + j] = o.stored;
            if (c_bf16) c_bf16[r * nout + j] = o.bf16;
            if (c_e4m3) c_e4m3[r * nout + j] = o.e4m3;
            ss += o.row_sq;
            rd += o.row_dot;
            if (o.amax > am || isnan(o.amax)) am = o.amax;
        }
        if (row_stat) row_stat[r] = has_row_dot ? rd : 1.0 / sqrt(ss / (double)nout + eps);
        if (amax_rows) amax_rows[r] = am;
        free(acc);
    }
    return bad ? -2 : 0;
}

int oracle_cols(const oracle_problem *p, const int64_t *cols, int64_t ncols,
                double *y, double *col_stat)
{
    oop ops[ORACLE_MAX_OPS];
    int nops;
    if (parse_program(p->program, ops, &nops)) return -1;
    int ip = find_pair(ops, nops);
    int ie = find_expand(ops, nops);
    int64_t nout = out_cols(p, ops, nops);
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = 0; c < ncols; ++c) {
        int64_t j = cols ? cols[c] : c;
        if (j < 0 || j >= nout) { bad = 1; continue; }
        double cs = 0.0;
        for (int64_t m = 0; m < p->M; ++m) {
            elem_out o;
            if (ie >= 0) {
                run_elem(p, ops, nops, m, j, acc_elem(p, m, expand_acc_col(j, ops[ie].i)), 0.0, &o);
            } else if (ip >= 0) {
                int64_t g = ops[ip].i;
                int64_t cg = (j / g) * 2 * g + j % g;
                run_elem(p, ops, nops, m, j, acc_elem(p, m, cg), acc_elem(p, m, cg + g), &o);
            } else {
                run_elem(p, ops, nops, m, j, acc_elem(p, m, j), 0.0, &o);
            }
            if (y) y[m * ncols + c] = o.stored;
            cs += o.col_v;
        }
        if (col_stat) col_stat[c] = cs;
    }
    return bad ? -2 : 0;
}

/* ------------------------------------------------------------------ */
/* RMSNorm backward (second pass)                                      */
/* ------------------------------------------------------------------ */

/* The gradient of y = x * S * w, S = (mean_n x^2 + eps)^(-1/2), written out:
 * dy/dx contributes S w dy directly and, through S, -x S^3 / N times
 * sum_n w dy x (dS/dx[n] = -S^3 x[n] / N).  "Lean4-TileLang Tensor Program
 * Superoptimizer", section 9 "RMSNorm" (the forward S and its row
 * broadcast), taken backward the way the CODA page's backward epilogues
 * pair an on-chip reduction with the output tile. */
void oracle_rmsnorm_backward(int64_t M, int64_t N, const uint16_t *dy, int64_t ld_dy,
                             const uint16_t *x, int64_t ld_x, const float *w, const float *s,
                             const double *r, const uint16_t *add, int64_t ld_add,
                             double *dx, double *dw)
{
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t m = 0; m < M; ++m) {
            double sm = (double)s[m];
            double c = sm * sm * sm * r[m] / (double)N;
            for (int64_t n = 0; n < N; ++n) {
                double wn = w ? (double)w[n] : 1.0;
                double g = wn * oracle_bf16_to_double(dy[m * ld_dy + n]);
                double v = sm * g - oracle_bf16_to_double(x[m * ld_x + n]) * c;
                if (add) v += oracle_bf16_to_double(add[m * ld_add + n]);
                dx[m * N + n] = v;
            }
        }
    }
    if (dw) {
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m)
                acc += oracle_bf16_to_double(dy[m * ld_dy + n]) * oracle_bf16_to_double(x[m * ld_x + n]) *
                       (double)s[m];
            dw[n] = acc;
        }
    }
}
