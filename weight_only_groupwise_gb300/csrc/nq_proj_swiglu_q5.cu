// Instantiation of the projection kernel: swiglu_q5.
#include "nq_launch.h"

namespace nq {
cudaError_t launch_proj_swiglu_q5(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    return launch_proj<5, true>(a, stream, pdl);
}
int cluster_capacity_swiglu_q5(int S, int smem) { return cluster_capacity_t<5, true>(S, smem); }
}  // namespace nq
