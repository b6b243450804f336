// Instantiations of the large-batch tensor-core projection kernel (nq_tc.cuh) for NVFP4
// weights, in their own translation unit so that the kernels compile in parallel.
#include "nq_launch.h"

namespace nq {
cudaError_t launch_tc_proj_fp4(const TcArgs& a, cudaStream_t stream, bool pdl) {
    switch (a.p.TP) {
        case 16: return tc_launch<kFp4, 16>(a, stream, pdl);
        case 32: return tc_launch<kFp4, 32>(a, stream, pdl);
        default: return tc_launch<kFp4, 64>(a, stream, pdl);
    }
}
}  // namespace nq
