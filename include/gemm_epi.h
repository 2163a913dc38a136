/*
 * gemm_epi.h -- C ABI of the GB300 (sm_103a) fused GEMM + epilogue engine.
 *
 * One call computes   acc = A @ B   (bf16 x bf16, or FP8 x FP8 with per-tensor
 * dequantisation factors, -> fp32 accumulate, on the tcgen05 tensor cores)
 * and, while each output tile is still on chip, runs a
 * short epilogue program on it: scaling, bias, row scale, residual add,
 * activations, a pairwise SwiGLU on interleaved gate/up columns, the GELU-tanh
 * derivative, AMAX, row RMS statistics, column sums, and bf16 / FP8-e4m3
 * stores.  Only the program's outputs reach global memory.
 *
 * Where the operations come from (page title, section):
 *  - GEMM O = X @ W with tiling, shared-memory staging, a pipelined K loop,
 *    swizzled tile order and tensor cores: "Lean4-TileLang Tensor Program
 *    Superoptimizer" (itsolotime.com), section 8 "Matmul"; and "Toi uu hoa GPU
 *    Kernel voi TileLang: Tu GEMM den FlashAttention" (aihot.vn), the tiled
 *    tensor-core GEMM paragraph.
 *  - bias + GELU applied to the register-resident accumulator before the
 *    final store: the TileLang tutorial, fused GEMM epilogue paragraph.
 *  - alpha given as a host scalar, bias, activation and an AMAX reduction in
 *    the same kernel for the next FP8 quantisation: "Huong dan su dung NVIDIA
 *    cuDNN Graph API" (aihot.vn), batched matmul epilogue paragraph.  The
 *    next GEMM of that FP8 loop reads the e4m3 output as an FP8 operand and
 *    multiplies the accumulator by the reciprocal of its scale (a_type,
 *    b_type, a_scale_inv, b_scale_inv).
 *  - SwiGLU out = up * silu(gate): Superoptimizer, section 7 "SwiGLU"; the
 *    RMSNorm-MLP's out = up * gate on rows scaled by S: section 10.
 *  - RMSNorm S = 1/sqrt(mean(x^2) + eps) and the row-broadcast rewrite
 *    (X*S)@W = (X@W)*S: Superoptimizer, sections 3 and 9 "RMSNorm"; its
 *    backward as a row reduction on the output tile plus a second pass
 *    (ROW_DOT, gemm_epi_rmsnorm_backward; CODA's backward epilogues).
 *  - a small set of composable epilogue primitives (scaling, reductions,
 *    pairwise transforms, accumulation) finished on the on-chip output tile,
 *    covering forward and backward work: "CODA: ... GEMM-Epilogue"
 *    (lehuy.net), "How CODA works".
 *  - create once (validate + plan), then execute with a pack of pointers and
 *    a caller-owned workspace: cuDNN Graph API tutorial, five-step build
 *    paragraph; launches are safe to capture in a CUDA graph (same page, CUDA
 *    graph paragraph).
 *
 * Memory and ownership
 *  - Every pointer in gemm_epi_args is a DEVICE pointer the caller allocated
 *    and owns (the workspace included).  The library owns only the host-side
 *    plan behind a gemm_epi_handle.
 *  - gemm_epi_run allocates nothing and never synchronises: it enqueues
 *    cudaMemsetAsync calls (reduction outputs and the workspace) and one
 *    kernel launch on `stream` (a cudaStream_t; NULL = legacy default stream).
 *  - Reduction outputs (amax, row_out, col_out) are OVERWRITTEN by each run,
 *    never accumulated across calls.
 *
 * Layouts (all row-major, strides in elements unless stated)
 *  - A: M x K of desc.a_type (bf16 by default), row stride lda >= K.
 *  - B: GEMM_EPI_B_KN: K x N of desc.b_type, row stride ldb >= N;
 *       GEMM_EPI_B_NK: N x K (B = W^T for a weight W stored N x K),
 *       row stride ldb >= K.  With GEMM_EPI_B_DUAL, B and B2 each hold N/2
 *       columns (K x N/2, or N/2 x K), both with row stride ldb.
 *  - FP8 operands (a_type and b_type both E4M3 or E5M2, in any mix) are one
 *    byte per element, so lda, ldb and their batch strides count bytes; B
 *    must be GEMM_EPI_B_NK (K contiguous, the usual N x K weight) and K a
 *    multiple of 16.
 *  - Output columns: N_out = N, N/2 after GEMM_EPI_OP_PAIR_SWIGLU / PAIR_MUL,
 *    2N after GEMM_EPI_OP_DSWIGLU.
 *  - C: M x N_out bf16, row stride ldc >= N_out.  C8: M x N_out e4m3 bytes,
 *    row stride ldc8 >= N_out (bytes).
 *  - residual / preact: M x N_out bf16, row stride ld_aux >= N_out (with
 *    DSWIGLU, preact holds the forward pre-activations, M x 2N).
 *  - bias: fp32, N_out values (N values when the op sits before the pair op).
 *  - row_scale: fp32, M values.  amax: 1 fp32.  row_out: M fp32.
 *    col_out: N_out fp32.
 *  - TMA needs every base pointer 16-byte aligned and every row stride a
 *    multiple of 16 bytes (8 bf16 elements, 16 e4m3 bytes); K must be a
 *    multiple of 8 (operand rows are read in whole 16-byte groups, so a
 *    ragged K tail would read the row padding); anything else is
 *    GEMM_EPI_ERR_MISALIGNED.  N and M need no alignment: outputs are written
 *    exactly within [0, M) x [0, N_out).  B with N % 8 != 0 may have the rest
 *    of its last 16-byte group read; those values never reach an output.
 *
 * Errors
 *  - create / run return synchronous validation errors and never launch
 *    anything when they fail; gemm_epi_last_error() gives a one-line reason
 *    (thread-local, valid until the next call on the same thread).
 *  - Every wait inside the kernel is bounded (timeout_ms).  A wait that runs
 *    out sets a status word in the workspace, the kernel drains what it has in
 *    flight, frees its tensor memory and returns; gemm_epi_query_status
 *    reports GEMM_EPI_ERR_TIMEOUT.  The kernel never traps.
 */
#ifndef GEMM_EPI_H
#define GEMM_EPI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_EPI_VERSION 1

/* The library is built with hidden symbol visibility: only these entry
 * points are exported, so several copies of it can share one process. */
#if defined(__GNUC__)
#define GEMM_EPI_API __attribute__((visibility("default")))
#else
#define GEMM_EPI_API
#endif

typedef enum gemm_epi_status {
    GEMM_EPI_OK = 0,
    GEMM_EPI_ERR_INVALID_VALUE = 1, /* bad size, NULL where required, bad program */
    GEMM_EPI_ERR_MISALIGNED = 2,    /* pointer or stride breaks the 16-byte TMA rule */
    GEMM_EPI_ERR_UNSUPPORTED = 3,   /* a legal program this library does not implement */
    GEMM_EPI_ERR_ARCH = 4,          /* current device is not compute capability 10.x */
    GEMM_EPI_ERR_CUDA = 5,          /* a CUDA runtime / driver call failed */
    GEMM_EPI_ERR_TIMEOUT = 6,       /* a bounded in-kernel wait ran out */
    GEMM_EPI_ERR_WORKSPACE = 7      /* workspace missing or smaller than required */
} gemm_epi_status;

/* Element types of the GEMM operands.  A and B are both BF16, or both 8-bit
 * (E4M3 and E5M2 may be mixed). */
typedef enum gemm_epi_type {
    GEMM_EPI_TYPE_BF16 = 0,
    GEMM_EPI_TYPE_E4M3 = 1,   /* OCP FP8 E4M3FN */
    GEMM_EPI_TYPE_E5M2 = 2    /* OCP FP8 E5M2 */
} gemm_epi_type;

typedef enum gemm_epi_b_layout {
    GEMM_EPI_B_KN = 0,   /* B stored K x N row-major (N contiguous) */
    GEMM_EPI_B_NK = 1,   /* B stored N x K row-major (K contiguous), i.e. W^T */
    /* Flag OR-ed onto KN or NK: two weight operands.  B and args.B2 each hold
     * N/2 columns (same layout and ldb); accumulator column n comes from B
     * column (n/256)*128 + n%128 when (n/128) is even and from B2's same
     * column when it is odd.  N % 256 == 0.  With a pair op of group 128 this
     * is out = f(X@B) * (X@B2): SwiGLU with separate W_gate (B) and W_up (B2)
     * sharing each A tile (Superoptimizer, section 7). */
    GEMM_EPI_B_DUAL = 16
} gemm_epi_b_layout;

/*
 * Epilogue primitives.  The program is applied per output element, in order,
 * to a running fp32 value y that starts as acc[m, n].  Element-wise ops
 * transform y; output ops (AMAX, STORE_BF16, STORE_E4M3, ROW_RMS_RSQRT,
 * ROW_DOT, COL_SUM) record y and leave it unchanged, and each appears at
 * most once per program (gemm_epi_create rejects a repeat with
 * GEMM_EPI_ERR_INVALID_VALUE).
 */
typedef enum gemm_epi_op_code {
    GEMM_EPI_OP_SCALE_ALPHA = 1,        /* y = alpha * y            (args.alpha)            */
    GEMM_EPI_OP_ADD_BIAS_COL = 2,       /* y = y + bias[n]          (args.bias)             */
    GEMM_EPI_OP_MUL_ROW_SCALE = 3,      /* y = y * row_scale[m]     (args.row_scale)        */
    GEMM_EPI_OP_ADD_RESIDUAL = 4,       /* y = y + residual[m, n]   (args.residual)         */
    GEMM_EPI_OP_ACT_GELU_TANH = 5,      /* y = gelu_tanh(y)                                 */
    GEMM_EPI_OP_ACT_RELU = 6,           /* y = max(y, 0)                                    */
    GEMM_EPI_OP_ACT_SILU = 7,           /* y = y * sigmoid(y)                               */
    GEMM_EPI_OP_PAIR_SWIGLU = 8,        /* y'[m,j] = silu(y[m,gate(j)]) * y[m,up(j)];
                                           i0 = group g in {1,2,4,8,16,32,128} (0 means 1):
                                           gate(j) = (j/g)*2g + j%g, up(j) = gate(j) + g;
                                           g = 1 is even = gate, odd = up.  N_out = N/2.  */
    GEMM_EPI_OP_MUL_GELU_TANH_GRAD = 9, /* y = y * gelu_tanh'(preact[m, n]) (args.preact)    */
    GEMM_EPI_OP_AMAX = 10,              /* *amax = max over valid (m,n) of |y|               */
    GEMM_EPI_OP_STORE_BF16 = 11,        /* C[m, n] = bf16_rne(y)                             */
    GEMM_EPI_OP_STORE_E4M3 = 12,        /* C8[m, n] = e4m3_rne_satfinite(y * args.fp8_scale) */
    GEMM_EPI_OP_ROW_RMS_RSQRT = 13,     /* row_out[m] = 1/sqrt(mean_n(v^2) + f0), f0 = eps;
                                           v = bf16_rne(y) when i0 == 0, v = y when i0 == 1 */
    GEMM_EPI_OP_COL_SUM = 14,           /* col_out[n] = sum over m of y                      */
    GEMM_EPI_OP_PAIR_MUL = 15,          /* y'[m,j] = y[m,gate(j)] * y[m,up(j)]: the RMSNorm-MLP's
                                           plain up * gate; same groups and N_out as
                                           PAIR_SWIGLU, at most one pair op per program      */
    GEMM_EPI_OP_DSWIGLU = 16,           /* backward of PAIR_SWIGLU: y[m,j] = dh for
                                           h = silu(gate) * up; gate = preact[m, gate(j)],
                                           up = preact[m, up(j)] (args.preact, the forward
                                           pre-activations, M x 2N); writes
                                           y'[m,gate(j)] = dh * up * silu'(gate),
                                           y'[m,up(j)] = dh * silu(gate);
                                           silu'(g) = s (1 + g (1 - s)), s = sigmoid(g).
                                           i0 = group g in {1,2,4,8,16} (0 means 1), same
                                           gate(j)/up(j) as PAIR_SWIGLU; N % g == 0;
                                           N_out = 2N.  Ops before it see the N accumulator
                                           columns, ops after it the 2N outputs; no other
                                           op may read preact or residual.  Counts as the
                                           program's pair op.                               */
    GEMM_EPI_OP_MUL_COL_SCALE = 17,     /* y = y * col_scale[n]     (args.col_scale)        */
    GEMM_EPI_OP_ROW_DOT = 18            /* row_out[m] = sum over n of y * residual[m, n]
                                           (args.residual): the row reduction of the
                                           RMSNorm backward, finished by
                                           gemm_epi_rmsnorm_backward.  Not with
                                           ROW_RMS_RSQRT (both write row_out).              */
} gemm_epi_op_code;

typedef struct gemm_epi_op {
    int32_t code; /* gemm_epi_op_code */
    int32_t i0;   /* integer argument (see the op) */
    float f0;     /* float argument (see the op) */
} gemm_epi_op;

#define GEMM_EPI_MAX_OPS 16

typedef struct gemm_epi_desc {
    int64_t M, N, K;          /* GEMM sizes; M, N >= 0; K >= 0, K % 8 == 0 (K % 16 == 0 for FP8
                                 operands; K == 0: acc = 0) */
    int64_t lda, ldb;         /* row strides of A and B, elements (bytes for FP8) */
    int64_t ldc;              /* row stride of C (bf16 elements); used with STORE_BF16 */
    int64_t ldc8;             /* row stride of C8 (bytes); used with STORE_E4M3 */
    int64_t ld_aux;           /* row stride of residual / preact (elements) */
    int32_t b_layout;         /* gemm_epi_b_layout */
    int32_t n_ops;            /* 0 .. GEMM_EPI_MAX_OPS */
    const gemm_epi_op *ops;   /* copied by gemm_epi_create */
    /* Batched GEMM (the cuDNN Graph API tutorial's batched matmul epilogue):
     * `batch` independent problems of the same shape and program; 0 or 1 is
     * one problem.  Strides between batches are in elements (bytes for C8);
     * 0 for A or B (and B2) shares that operand across the batch.  Per batch:
     * row_scale, row_out (M values each) and col_out (N_out each) advance by
     * M and N_out; bias is shared; AMAX is one value over the whole batch. */
    int64_t batch;
    int64_t batch_stride_a, batch_stride_b, batch_stride_c, batch_stride_c8, batch_stride_aux;
    int32_t a_type, b_type;   /* gemm_epi_type of A and of B (and B2); 0 = BF16 */
} gemm_epi_desc;

typedef struct gemm_epi_args {
    const void *A;            /* desc.a_type, device */
    const void *B;            /* desc.b_type, device */
    float alpha;              /* SCALE_ALPHA */
    float fp8_scale;          /* STORE_E4M3 */
    const float *bias;        /* ADD_BIAS_COL */
    const float *row_scale;   /* MUL_ROW_SCALE */
    const void *residual;     /* ADD_RESIDUAL, bf16 */
    const void *preact;       /* MUL_GELU_TANH_GRAD, bf16 */
    void *C;                  /* STORE_BF16 output */
    void *C8;                 /* STORE_E4M3 output */
    float *amax;              /* AMAX output, 1 value */
    float *row_out;           /* ROW_RMS_RSQRT output, M values */
    float *col_out;           /* COL_SUM output, N_out values */
    void *workspace;          /* gemm_epi_workspace_size(h) bytes, 16-byte aligned */
    size_t workspace_bytes;
    uint32_t timeout_ms;      /* bound of every in-kernel wait; 0 = 2000 ms */
    uint32_t debug_flags;     /* 0 in normal use; GEMM_EPI_DEBUG_* for tests */
    const void *B2;           /* second weight operand with GEMM_EPI_B_DUAL, B's type */
    /* Per-tensor dequantisation factors, device fp32 scalars or NULL (= 1):
     * the accumulator the program starts from is
     * (*a_scale_inv) * (*b_scale_inv) * (A @ B), the product taken in fp32.
     * For an FP8 operand quantised as code = fp8(x * s) this is 1/s; reading
     * it from device memory lets a scale derived from a previous AMAX feed
     * the next GEMM without a host round trip.  Any operand type. */
    const float *a_scale_inv;
    const float *b_scale_inv;
    const float *col_scale;   /* MUL_COL_SCALE: fp32, one value per column at its point of use */
} gemm_epi_args;

/* Test hook: the first CTA's producer skips the operand loads of the first
 * pipeline stage of its first tile (two K-blocks on the CTA-pair loop, one
 * on the single-CTA loop) and never arms that stage's full barrier, so that
 * the MMA warp's bounded wait runs out. */
#define GEMM_EPI_DEBUG_SKIP_FIRST_LOAD 1u
/* Test hook: as above, but only the first tile's second K-block is not
 * loaded.  On the CTA-pair loop it shares a stage with the first, whose
 * barrier is then armed and stays short of those bytes: the abort path
 * settles a partly loaded stage.  On the single-CTA loop it is a stage of
 * its own, never armed. */
#define GEMM_EPI_DEBUG_SKIP_SECOND_LOAD 16u
/* Test hooks: run the 1-SM main loop (one CTA per 128 x 256 tile) or the
 * 2-SM one (a CTA pair per 256 x 256 tile) whatever M is.  By default the
 * 2-SM loop runs when M > 128. */
#define GEMM_EPI_DEBUG_FORCE_1SM 2u
#define GEMM_EPI_DEBUG_FORCE_2SM 4u
/* Test hook: run the op-interpreting kernel even when the program has a
 * compiled (static) kernel, so both forms can be checked on one program. */
#define GEMM_EPI_DEBUG_FORCE_INTERPRETER 8u

typedef struct gemm_epi_plan *gemm_epi_handle;

/* Validates the descriptor and builds a host-side plan.  Pure host code: no
 * CUDA call, no device needed.  *out is set only on GEMM_EPI_OK. */
GEMM_EPI_API gemm_epi_status gemm_epi_create(gemm_epi_handle *out, const gemm_epi_desc *desc);

/* Frees the plan.  NULL is accepted. */
GEMM_EPI_API gemm_epi_status gemm_epi_destroy(gemm_epi_handle h);

/* Bytes of device workspace gemm_epi_run needs for this plan (>= 256). */
GEMM_EPI_API size_t gemm_epi_workspace_size(gemm_epi_handle h);

/* Output columns of the plan (N, N/2 after a pair op, 2N after DSWIGLU); -1 for NULL. */
GEMM_EPI_API int64_t gemm_epi_out_cols(gemm_epi_handle h);

/* Enqueues the fused kernel on `stream`.  Checks the device (compute
 * capability 10.x), every pointer the program uses (non-NULL, 16-byte
 * aligned) and the workspace.  Asynchronous; capture-safe. */
GEMM_EPI_API gemm_epi_status gemm_epi_run(gemm_epi_handle h, const gemm_epi_args *args, void *stream);

/* The unfused baseline with the same semantics: a bare GEMM into `scratch`
 * (M x N bf16 pre-epilogue accumulator, row stride ld_scratch >= N, caller
 * owned), then a separate memory-bound epilogue pass that reads it back.  The
 * accumulator is rounded to bf16 between the two, so results differ from the
 * fused path by that rounding.  For measurement only. */
GEMM_EPI_API gemm_epi_status gemm_epi_run_unfused(gemm_epi_handle h, const gemm_epi_args *args,
                                     void *scratch, int64_t ld_scratch, void *stream);

/* Allocation-free variant of gemm_epi_run.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory --
 * code running inside a host framework or plugin interface that hands it
 * only input and output pointers and owns every other allocation, or a
 * latency-critical loop that must not pay for cudaMalloc's implicit device
 * synchronisation -- and so have no way to supply a workspace.
 *  - Same arguments and semantics as gemm_epi_run; args->workspace and
 *    args->workspace_bytes are ignored.  Nothing is allocated: no cudaMalloc,
 *    cudaFree or allocating library routine is called.
 *  - The scratch (status words and per-row-tile counters) is one static
 *    device array of GEMM_EPI_NO_ALLOC_SCRATCH_BYTES bytes inside the
 *    library; every GPU that loads the library keeps it until the process
 *    exits.  Plans whose gemm_epi_workspace_size exceeds it are rejected
 *    with GEMM_EPI_ERR_WORKSPACE: after 256 bytes of status words it holds
 *    16,320 row-block counters, and a plan needs ceil(M/256) * 2 * batch of
 *    them (M up to 2,088,960 rows for one problem, a batch-th of that for a
 *    batch).
 *  - The first call on a device looks up the array's address on that device
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - All calls share the array and clear it on their stream before the
 *    kernel; calls whose kernels overlap on the GPU (several streams, several
 *    host threads) race on it and must be serialised by the caller.
 *  - A timed-out in-kernel wait is recorded in that array and is not
 *    reported back; use gemm_epi_run with a workspace and
 *    gemm_epi_query_status when the status is needed. */
#define GEMM_EPI_NO_ALLOC_SCRATCH_BYTES 65536
GEMM_EPI_API gemm_epi_status gemm_epi_run_no_alloc(gemm_epi_handle h, const gemm_epi_args *args, void *stream);

/*
 * RMSNorm backward, second pass.  For y = x * S * w (S[m] = 1/sqrt(mean_n
 * x^2 + eps), the forward's ROW_RMS_RSQRT output) and the upstream gradient
 * dy (the C of a GEMM whose program ran MUL_COL_SCALE(w) and ROW_DOT with
 * residual = x after storing dy):
 *   dx[m,n] = S[m] w[n] dy[m,n] - x[m,n] S[m]^3 r[m] / N  (+ add[m,n])
 *   dw[n]   = sum over m of dy[m,n] x[m,n] S[m]
 * with r = the ROW_DOT output.  The per-row reduction spans every column of
 * the row, so this step follows the GEMM as its own memory-bound kernel
 * (reads dy, x and add once, writes dx once).  dy, x, add, dx: bf16 row-major,
 * 16-byte aligned, row strides multiples of 8 elements.  w NULL means 1; add
 * NULL means none; dx or dw may be NULL (not computed); dw is overwritten.
 */
typedef struct gemm_epi_rmsnorm_bwd_args {
    int64_t M, N;
    const void *dy;  int64_t ld_dy;
    const void *x;   int64_t ld_x;
    const void *add; int64_t ld_add;
    const float *w;  /* N values */
    const float *s;  /* M values */
    const float *r;  /* M values */
    void *dx;        int64_t ld_dx;
    float *dw;       /* N values */
} gemm_epi_rmsnorm_bwd_args;

/* Enqueues the second pass on `stream` (a cudaStream_t).  Asynchronous;
 * capture-safe; checks sizes, pointers and alignment first. */
GEMM_EPI_API gemm_epi_status gemm_epi_rmsnorm_backward(const gemm_epi_rmsnorm_bwd_args *args, void *stream);

/* Synchronises `stream`, then reads the status words the last run on that
 * workspace left: GEMM_EPI_OK or GEMM_EPI_ERR_TIMEOUT (the last-error string
 * then names the wait and the block).  For diagnostics, the first four
 * 32-bit words of the workspace hold: [0] bit 0 an in-kernel wait ran out,
 * bit 1 the bounded wait for the operand loads still in flight after it
 * also ran out; [1] which wait; [2] the block; [3] the pipeline stages whose
 * loads the abort path settled (bits 0-7: a stage with K-blocks that were
 * never loaded, bits 8-15: a phase the even CTA of a pair had not armed). */
GEMM_EPI_API gemm_epi_status gemm_epi_query_status(gemm_epi_handle h, const void *workspace, void *stream);

/* Static description of a status code. */
GEMM_EPI_API const char *gemm_epi_status_string(gemm_epi_status s);

/* One-line reason for the most recent failure on this thread ("" if none). */
GEMM_EPI_API const char *gemm_epi_last_error(void);

/* GEMM_EPI_VERSION of the loaded library. */
GEMM_EPI_API int gemm_epi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_EPI_H */
