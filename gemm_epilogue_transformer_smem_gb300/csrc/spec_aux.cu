// spec_aux.cu -- static kernels of the FP8, residual + row RMS, GELU backward
// and SwiGLU backward programs (compiled apart from the others to keep builds
// parallel).
#include "programs.cuh"

namespace ge {

const KernelSpec kSpecsAux[] = {
    make_spec<ProgFp8>("relu_amax_fp8"),
    make_spec<ProgResidualRms>("residual_row_rms"),
    make_spec<ProgGeluGradColSum>("gelu_grad_col_sum"),
    make_spec<ProgDSwiGLU>("dswiglu"),
};
const int kNumSpecsAux = sizeof(kSpecsAux) / sizeof(kSpecsAux[0]);

}  // namespace ge
