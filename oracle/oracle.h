/*
 * oracle.h -- fp64 CPU reference of the fused GEMM + epilogue.
 *
 * TEST INFRASTRUCTURE ONLY: used by tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py.  Shares nothing with the CUDA
 * library.  See oracle.c for the definition and its sources.
 */
#ifndef GEMM_EPI_ORACLE_H
#define GEMM_EPI_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int64_t M, N, K;
    int b_is_nk;                 /* 0: B is K x N row-major; 1: B is N x K row-major */
    const void *A;               /* M x K elements of type a_type, row stride lda */
    int64_t lda;
    const void *B;               /* elements of type b_type */
    int64_t ldb;
    const void *B2;              /* second weight operand or NULL (same layout, ldb) */
    double alpha;                /* op "alpha" */
    const float *bias;           /* op "bias": one value per column at its point of use */
    const float *row_scale;      /* op "row_scale": M values */
    const uint16_t *residual;    /* op "residual": bf16, M x (columns), row stride ld_aux */
    const uint16_t *preact;      /* ops "gelu_tanh_grad" (M x columns) and "dswiglu"
                                    (M x 2N forward gate/up pairs): bf16, stride ld_aux */
    int64_t ld_aux;
    double fp8_scale;            /* op "store_e4m3": code = e4m3(value * fp8_scale) */
    const char *program;         /* comma-separated op names, optional ":arg" */
    int a_type, b_type;          /* ORACLE_BF16 (bit patterns), ORACLE_E4M3, ORACLE_E5M2 (codes) */
    double a_scale_inv;          /* the accumulator is a_scale_inv * b_scale_inv * (A @ B) */
    double b_scale_inv;          /* (1.0 for unscaled operands) */
    const float *col_scale;      /* op "col_scale": one value per column at its point of use */
} oracle_problem;

enum { ORACLE_BF16 = 0, ORACLE_E4M3 = 1, ORACLE_E5M2 = 2 };

/* Whole output rows for the listed row indices (rows == NULL: rows 0..nrows-1).
 * Every output pointer may be NULL.  y: value at store_bf16 (or final value),
 * nrows x out_cols.  Returns 0, -1 for a bad program, -2 for a bad index. */
int oracle_rows(const oracle_problem *p, const int64_t *rows, int64_t nrows,
                double *y, uint16_t *c_bf16, uint8_t *c_e4m3, double *row_stat,
                double *amax_rows);

/* Whole output columns (all M rows) for the listed columns.  y: M x ncols. */
int oracle_cols(const oracle_problem *p, const int64_t *cols, int64_t ncols,
                double *y, double *col_stat);

int oracle_out_cols(const oracle_problem *p);

/* RMSNorm backward, finished from the row reduction: for y = x * S * w with
 * S[m] = 1/sqrt(mean_n x^2 + eps) and upstream gradient dy,
 *   dx[m,n] = S[m] w[n] dy[m,n] - x[m,n] S[m]^3 r[m] / N (+ add[m,n]),
 *   r[m]    = sum_n w[n] dy[m,n] x[m,n]           (given),
 *   dw[n]   = sum_m dy[m,n] x[m,n] S[m].
 * dy, x, add: bf16 bit patterns with row strides; w NULL means 1; add NULL
 * means none; dx (M x N) and dw (N) in fp64, either may be NULL. */
void oracle_rmsnorm_backward(int64_t M, int64_t N, const uint16_t *dy, int64_t ld_dy,
                             const uint16_t *x, int64_t ld_x, const float *w, const float *s,
                             const double *r, const uint16_t *add, int64_t ld_add,
                             double *dx, double *dw);

double oracle_bf16_to_double(uint16_t bits);
uint16_t oracle_double_to_bf16(double x);
uint8_t oracle_double_to_e4m3(double x);
double oracle_e4m3_to_double(uint8_t c);
double oracle_e5m2_to_double(uint8_t c);
double oracle_gelu_tanh(double x);
double oracle_gelu_tanh_grad(double x);
double oracle_silu(double x);
double oracle_silu_grad(double x);

#ifdef __cplusplus
}
#endif

#endif
