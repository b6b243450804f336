// Instantiation of the projection kernel: SwiGLU blocks with NVFP4 gate and up weights
// (fp16 operands).
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_swiglu_fp4(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj_f16_only<kFp4, true>(a, stream, pdl);
}
}  // namespace nq
