// Instantiation of the projection kernel: swiglu_q5.
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_swiglu_q5(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj<5, true>(a, stream, pdl);
}
}  // namespace nq
