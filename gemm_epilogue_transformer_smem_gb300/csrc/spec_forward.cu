// spec_forward.cu -- static kernels of the bare GEMM, bias + GELU + AMAX,
// SwiGLU and RMSNorm-consuming programs (compiled apart from the others to
// keep builds parallel).
#include "programs.cuh"

namespace ge {

const KernelSpec kSpecsForward[] = {
    make_spec<ProgBare>("bare"),
    make_spec<ProgBiasGelu>("bias_gelu_amax"),
    make_spec<ProgSwiGLU>("swiglu"),
    make_spec<ProgRmsSwiGLU>("row_scale_swiglu"),
    make_spec<ProgRmsGlu>("row_scale_pair_mul"),
    make_spec<ProgSwiGLU2W>("swiglu_two_weights"),
    make_spec<ProgRmsSwiGLU2W>("row_scale_swiglu_two_weights"),
    make_spec<ProgRmsGlu2W>("row_scale_pair_mul_two_weights"),
};
const int kNumSpecsForward = sizeof(kSpecsForward) / sizeof(kSpecsForward[0]);

}  // namespace ge
