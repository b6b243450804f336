// Instantiation of the projection kernel: swiglu_q4.
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_swiglu_q4(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj<4, true>(a, stream, pdl);
}
int cluster_capacity_swiglu_q4(int S, int smem) { return cluster_capacity_t<4, true>(S, smem); }
}  // namespace nq
