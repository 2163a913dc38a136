// spec_forward.cu -- static kernels of the bare GEMM, bias + GELU + AMAX and
// SwiGLU programs (compiled apart from the others to keep builds parallel).
#include "programs.cuh"

namespace ge {

const KernelSpec kSpecsForward[] = {
    make_spec<ProgBare>("bare"),
    make_spec<ProgBiasGelu>("bias_gelu_amax"),
    make_spec<ProgSwiGLU>("swiglu"),
};
const int kNumSpecsForward = sizeof(kSpecsForward) / sizeof(kSpecsForward[0]);

}  // namespace ge
