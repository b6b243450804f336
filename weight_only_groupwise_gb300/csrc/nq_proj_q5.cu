// Instantiation of the projection kernel: q5.
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_q5(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj<5, false>(a, stream, pdl);
}
int cluster_capacity_q5(int S, int smem) { return cluster_capacity_t<5, false>(S, smem); }
}  // namespace nq
