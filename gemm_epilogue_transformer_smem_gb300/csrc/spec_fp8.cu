// spec_fp8.cu -- kernels for 8-bit (e4m3 / e5m2) operands: the interpreting
// kernel and static forms of the programs an FP8 GEMM is most often given
// (compiled apart from the bf16 kernels to keep builds parallel).
#include "programs.cuh"

namespace ge {

const KernelSpec kSpecsFp8[] = {
    make_spec<ProgBare, 1>("bare_fp8"),
    make_spec<ProgFp8, 1>("relu_amax_fp8_fp8"),
    make_spec<ProgBiasGelu, 1>("bias_gelu_amax_fp8"),
    make_spec<ProgSwiGLU, 1>("swiglu_fp8"),
    make_spec<ProgSwiGLU2W, 1>("swiglu_two_weights_fp8"),
};
const int kNumSpecsFp8 = sizeof(kSpecsFp8) / sizeof(kSpecsFp8[0]);

const void* const kDynamicFp8[2] = {
    reinterpret_cast<const void*>(&fused_gemm_epilogue_kernel<1, DynamicProgram, 1>),
    reinterpret_cast<const void*>(&fused_gemm_epilogue_kernel<2, DynamicProgram, 1>)};

}  // namespace ge
