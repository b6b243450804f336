// Instantiations and host launch of the large-batch tensor-core projection kernel (nq_tc.cuh):
// the activation tensor map and the launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "nq_launch.h"

namespace nq {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

template <int BITS, int TP>
cudaError_t launch_t(const TcArgs& a, cudaStream_t stream, bool pdl) {
    auto kern = tc_proj_kernel<BITS, TP>;
    static thread_local int set_for_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (set_for_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        set_for_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.p.P);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = a.p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

// X (bf16 [T][K], row-major) as a 3-D tensor [K/8][T][8]: a box {8, TP, 32} lands in shared
// memory as K-major core matrices (8 tokens x 8 K), core (token block n8, K block k8) at byte
// 128 n8 + 16 TP k8; tokens T..TP-1 are outside the tensor and read as zeros.
bool encode_x_map(CUtensorMap* map, const void* X, int T, int K, int TP) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {8, (cuuint64_t)T, (cuuint64_t)(K / 8)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 16};
    const cuuint32_t box[3] = {8, (cuuint32_t)TP, (cuuint32_t)(kTcStageGroups * kGroup / 8)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(X), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_tc_proj(int bits, const TcArgs& a, cudaStream_t stream, bool pdl) {
    switch (a.p.TP) {
        case 16: return bits == 4 ? launch_t<4, 16>(a, stream, pdl) : launch_t<5, 16>(a, stream, pdl);
        case 32: return bits == 4 ? launch_t<4, 32>(a, stream, pdl) : launch_t<5, 32>(a, stream, pdl);
        default: return bits == 4 ? launch_t<4, 64>(a, stream, pdl) : launch_t<5, 64>(a, stream, pdl);
    }
}

}  // namespace nq
