// programs.cuh -- the epilogue programs compiled as static kernels.
//
// gemm_epi_create matches a plan's op list against these entries (codes and
// pair group, in order); a match launches the static kernel, anything else
// the interpreting one.  Per-call values (alpha, bias, eps, scales, ...) are
// runtime arguments either way.
#pragma once

#include "fused_kernel.cuh"
#include "unfused_kernel.cuh"

namespace ge {

constexpr int PAIR_G1 = GEMM_EPI_OP_PAIR_SWIGLU | (1 << 8);
constexpr int PAIR_MUL_G1 = GEMM_EPI_OP_PAIR_MUL | (1 << 8);
constexpr int PAIR_G128 = GEMM_EPI_OP_PAIR_SWIGLU | (128 << 8);
constexpr int PAIR_MUL_G128 = GEMM_EPI_OP_PAIR_MUL | (128 << 8);

// Bare GEMM: the store-only epilogue (also the first half of the unfused path).
using ProgBare = StaticProgram<GEMM_EPI_OP_STORE_BF16>;
// gelu_tanh(alpha * acc + bias), AMAX, bf16 store.
using ProgBiasGelu = StaticProgram<GEMM_EPI_OP_SCALE_ALPHA, GEMM_EPI_OP_ADD_BIAS_COL, GEMM_EPI_OP_ACT_GELU_TANH,
                                   GEMM_EPI_OP_AMAX, GEMM_EPI_OP_STORE_BF16>;
// silu(gate) * up on even/odd columns, bf16 store.
using ProgSwiGLU = StaticProgram<PAIR_G1, GEMM_EPI_OP_STORE_BF16>;
// RMSNorm-consuming up-projections: rows scaled by the previous layer's S,
// then silu(gate) * up or the plain gate * up, bf16 store.
using ProgRmsSwiGLU = StaticProgram<GEMM_EPI_OP_MUL_ROW_SCALE, PAIR_G1, GEMM_EPI_OP_STORE_BF16>;
using ProgRmsGlu = StaticProgram<GEMM_EPI_OP_MUL_ROW_SCALE, PAIR_MUL_G1, GEMM_EPI_OP_STORE_BF16>;
// The same with separate gate / up weights (GEMM_EPI_B_DUAL, pair group 128).
using ProgSwiGLU2W = StaticProgram<PAIR_G128, GEMM_EPI_OP_STORE_BF16>;
using ProgRmsSwiGLU2W = StaticProgram<GEMM_EPI_OP_MUL_ROW_SCALE, PAIR_G128, GEMM_EPI_OP_STORE_BF16>;
using ProgRmsGlu2W = StaticProgram<GEMM_EPI_OP_MUL_ROW_SCALE, PAIR_MUL_G128, GEMM_EPI_OP_STORE_BF16>;
// relu(alpha * acc + bias), AMAX, bf16 and e4m3 stores.
using ProgFp8 = StaticProgram<GEMM_EPI_OP_SCALE_ALPHA, GEMM_EPI_OP_ADD_BIAS_COL, GEMM_EPI_OP_ACT_RELU,
                              GEMM_EPI_OP_AMAX, GEMM_EPI_OP_STORE_BF16, GEMM_EPI_OP_STORE_E4M3>;
// residual + acc, bf16 store, per-row rsqrt(mean square + eps).
using ProgResidualRms = StaticProgram<GEMM_EPI_OP_ADD_RESIDUAL, GEMM_EPI_OP_STORE_BF16,
                                      GEMM_EPI_OP_ROW_RMS_RSQRT>;
// SwiGLU backward: both gradients from dh and the forward gate / up pairs.
constexpr int DSWIGLU_G1 = GEMM_EPI_OP_DSWIGLU | (1 << 8);
using ProgDSwiGLU = StaticProgram<DSWIGLU_G1, GEMM_EPI_OP_STORE_BF16>;
// RMSNorm backward, first pass: store dy, scale by the norm weight, reduce
// against the RMSNorm input per row.
using ProgRmsBwd = StaticProgram<GEMM_EPI_OP_STORE_BF16, GEMM_EPI_OP_MUL_COL_SCALE, GEMM_EPI_OP_ROW_DOT>;
// acc * gelu_tanh'(preact), bf16 store, column sums.
using ProgGeluGradColSum = StaticProgram<GEMM_EPI_OP_MUL_GELU_TANH_GRAD, GEMM_EPI_OP_STORE_BF16,
                                         GEMM_EPI_OP_COL_SUM>;

// Common forward / backward programs outside the benchmark set.
using ProgBias = StaticProgram<GEMM_EPI_OP_ADD_BIAS_COL, GEMM_EPI_OP_STORE_BF16>;
using ProgBiasGeluNoAmax = StaticProgram<GEMM_EPI_OP_ADD_BIAS_COL, GEMM_EPI_OP_ACT_GELU_TANH, GEMM_EPI_OP_STORE_BF16>;
using ProgBiasRelu = StaticProgram<GEMM_EPI_OP_ADD_BIAS_COL, GEMM_EPI_OP_ACT_RELU, GEMM_EPI_OP_STORE_BF16>;
using ProgBiasSilu = StaticProgram<GEMM_EPI_OP_ADD_BIAS_COL, GEMM_EPI_OP_ACT_SILU, GEMM_EPI_OP_STORE_BF16>;
using ProgAlphaBiasGelu = StaticProgram<GEMM_EPI_OP_SCALE_ALPHA, GEMM_EPI_OP_ADD_BIAS_COL, GEMM_EPI_OP_ACT_GELU_TANH,
                                        GEMM_EPI_OP_STORE_BF16>;
using ProgResidual = StaticProgram<GEMM_EPI_OP_ADD_RESIDUAL, GEMM_EPI_OP_STORE_BF16>;
using ProgGeluGrad = StaticProgram<GEMM_EPI_OP_MUL_GELU_TANH_GRAD, GEMM_EPI_OP_STORE_BF16>;
using ProgAlpha = StaticProgram<GEMM_EPI_OP_SCALE_ALPHA, GEMM_EPI_OP_STORE_BF16>;
using ProgRowScale = StaticProgram<GEMM_EPI_OP_MUL_ROW_SCALE, GEMM_EPI_OP_STORE_BF16>;

// One compiled program: its op list (code | pair group << 8), the operand
// width it was compiled for, its kernels for the 1-SM and 2-SM main loops and
// its separate-pass kernel for the unfused baseline (NULL if the pass does
// not cover the program).
struct KernelSpec {
  const char* name;
  int n_ops;
  int ops[GEMM_EPI_MAX_OPS];
  int in8;  // 1: 8-bit operands
  const void* kernel_1sm;
  const void* kernel_2sm;
  const void* kernel_unfused;
};

template <class Prog, int IN8, int... Is>
inline KernelSpec make_spec(const char* name, std::integer_sequence<int, Is...>) {
  return KernelSpec{name,
                    Prog::n,
                    {(Prog::code_of(Is) | (Prog::arg_of(Is) << 8))...},
                    IN8,
                    reinterpret_cast<const void*>(&fused_gemm_epilogue_kernel<1, Prog, IN8>),
                    reinterpret_cast<const void*>(&fused_gemm_epilogue_kernel<2, Prog, IN8>),
                    unfused_kernel_for<Prog>()};
}

template <class Prog, int IN8 = 0>
inline KernelSpec make_spec(const char* name) {
  return make_spec<Prog, IN8>(name, std::make_integer_sequence<int, Prog::n>{});
}

// Tables defined by the translation units that instantiate the kernels.
extern const KernelSpec kSpecsForward[];
extern const int kNumSpecsForward;
extern const KernelSpec kSpecsAux[];
extern const int kNumSpecsAux;
extern const KernelSpec kSpecsFp8[];
extern const int kNumSpecsFp8;
extern const KernelSpec kSpecsCommon[];
extern const int kNumSpecsCommon;
// The interpreting kernels for 8-bit operands (1-SM, 2-SM), from the same
// translation unit as kSpecsFp8.
extern const void* const kDynamicFp8[2];

}  // namespace ge
