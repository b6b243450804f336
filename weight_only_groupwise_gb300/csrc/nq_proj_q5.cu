// Instantiation of the projection kernel: q5.
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_q5(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj<5, false>(a, stream, pdl);
}
}  // namespace nq
