// Instantiation of the projection kernel: q4.
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_q4(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj<4, false>(a, stream, pdl);
}
int cluster_capacity_q4(int S, int smem) { return cluster_capacity_t<4, false>(S, smem); }
}  // namespace nq
