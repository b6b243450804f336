// Instantiation of the projection kernel: swiglu_q4.
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_swiglu_q4(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj<4, true>(a, stream, pdl);
}
}  // namespace nq
