// spec_common.cu -- static kernels of common forward and backward programs
// outside the benchmark set (a linear layer with bias, bias + activation,
// the residual add, the GELU derivative without column sums, plain scales),
// so that they skip the interpreter.  Compiled apart from the others to keep
// builds parallel.
#include "programs.cuh"

namespace ge {

const KernelSpec kSpecsCommon[] = {
    make_spec<ProgBias>("bias"),
    make_spec<ProgBiasGeluNoAmax>("bias_gelu"),
    make_spec<ProgBiasRelu>("bias_relu"),
    make_spec<ProgBiasSilu>("bias_silu"),
    make_spec<ProgAlphaBiasGelu>("alpha_bias_gelu"),
    make_spec<ProgResidual>("residual"),
    make_spec<ProgGeluGrad>("gelu_grad"),
    make_spec<ProgAlpha>("alpha"),
    make_spec<ProgRowScale>("row_scale"),
};
const int kNumSpecsCommon = sizeof(kSpecsCommon) / sizeof(kSpecsCommon[0]);

}  // namespace ge
