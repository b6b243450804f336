// Instantiations of the large-batch tensor-core projection kernel (nq_tc.cuh) that finish a
// SwiGLU block: the gate projection (fp32 G) and the up projection (bf16 silu(G) * U), in their
// own translation unit so that the kernels compile in parallel.
#include "nq_launch.h"

namespace nq {
namespace {
template <int BITS, int MODE>
cudaError_t launch_tp(const TcArgs& a, cudaStream_t stream, bool pdl) {
    switch (a.p.TP) {
        case 16: return tc_launch<BITS, 16, MODE>(a, stream, pdl);
        case 32: return tc_launch<BITS, 32, MODE>(a, stream, pdl);
        default: return tc_launch<BITS, 64, MODE>(a, stream, pdl);
    }
}

template <int MODE>
cudaError_t launch_mode(int bits, const TcArgs& a, cudaStream_t stream, bool pdl) {
    if (bits == 4) return launch_tp<4, MODE>(a, stream, pdl);
    if (bits == 5) return launch_tp<5, MODE>(a, stream, pdl);
    return launch_tp<kFp4, MODE>(a, stream, pdl);
}
}  // namespace

cudaError_t launch_tc_proj_swiglu(int bits, int mode, const TcArgs& a, cudaStream_t stream, bool pdl) {
    return mode == kTcOutGate ? launch_mode<kTcOutGate>(bits, a, stream, pdl)
                              : launch_mode<kTcOutSwiglu>(bits, a, stream, pdl);
}
}  // namespace nq
