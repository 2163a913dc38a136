// spec_aux.cu -- static kernels of the FP8, residual + row RMS, GELU backward,
// SwiGLU backward and RMSNorm backward programs (compiled apart from the
// others to keep builds parallel).
#include "programs.cuh"

namespace ge {

const KernelSpec kSpecsAux[] = {
    make_spec<ProgFp8>("relu_amax_fp8"),
    make_spec<ProgResidualRms>("residual_row_rms"),
    make_spec<ProgGeluGradColSum>("gelu_grad_col_sum"),
    make_spec<ProgDSwiGLU>("dswiglu"),
    make_spec<ProgRmsBwd>("rmsnorm_backward_dy"),
};
const int kNumSpecsAux = sizeof(kSpecsAux) / sizeof(kSpecsAux[0]);

}  // namespace ge
