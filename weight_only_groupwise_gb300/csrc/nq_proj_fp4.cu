// Instantiation of the projection kernel: NVFP4 weights (fp16 operands).
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_fp4(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj_f16_only<kFp4>(a, stream, pdl);
}
}  // namespace nq
