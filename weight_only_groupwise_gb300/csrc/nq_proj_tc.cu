// Instantiations (4- and 5-bit codes) and host side of the large-batch tensor-core projection
// kernel (nq_tc.cuh): the tensor maps and the launch.
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

}  // namespace

bool tensor_maps_available() { return encode_fn() != nullptr; }

// X (bf16 [T][K], row-major) as a 3-D tensor [K/64][T][64]: a box {64, TP, BG} (BG = the
// stage's groups) lands in shared memory as one [TP][64] block per group, 128-byte rows with
// the 128-byte swizzle (16-byte chunk c of token t at chunk c ^ (t % 8)), which is the tensor
// core's K-major swizzled layout; tokens T..TP-1 are outside the tensor and read as zeros.
// 128-byte rows keep the copy engine's request count at TP per group.
bool encode_x_map(CUtensorMap* map, const void* X, int T, int K, int TP) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kGroup, (cuuint64_t)T, (cuuint64_t)(K / kGroup)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)kGroup * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kGroup, (cuuint32_t)TP, (cuuint32_t)tc_stage_groups(TP)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(X), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The packed codes and scales of a matrix as 3-D tensors of 8-byte elements [RT][G][bytes / 8]
// (16-row tiles, 64-wide K groups, one tile-group block): a box {bytes / 8, BG, kTcTiles} (BG =
// the stage's groups for TP padded tokens) is one stage's codes (or scales) of a 128-row
// block, laid out tile-major as the kernel reads them; tiles past RT and groups past G read as
// zeros.
bool encode_weight_maps(CUtensorMap* wmap, CUtensorMap* smap, const void* W, const void* S, int bits, int K, int N,
                        int TP) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int G = K / kGroup, RT = N / kTileRows;
    const cuuint32_t estr[3] = {1, 1, 1};
    const int tb = code_tile_bytes(bits);
    const cuuint64_t wdims[3] = {(cuuint64_t)(tb / 8), (cuuint64_t)G, (cuuint64_t)RT};
    const cuuint64_t wstr[2] = {(cuuint64_t)tb, (cuuint64_t)G * tb};
    const cuuint32_t bg = (cuuint32_t)tc_stage_groups(TP);
    const cuuint32_t wbox[3] = {(cuuint32_t)(tb / 8), bg, (cuuint32_t)kTcTiles};
    const int stb = scale_tile_bytes(bits);
    const cuuint64_t sdims[3] = {(cuuint64_t)(stb / 8), (cuuint64_t)G, (cuuint64_t)RT};
    const cuuint64_t sstr[2] = {(cuuint64_t)stb, (cuuint64_t)G * stb};
    const cuuint32_t sbox[3] = {(cuuint32_t)(stb / 8), bg, (cuuint32_t)kTcTiles};
    return fn(wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void*>(W), wdims, wstr, wbox, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
           fn(smap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void*>(S), sdims, sstr, sbox, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_tc_proj(int bits, const TcArgs& a, cudaStream_t stream, bool pdl) {
    if (bits == kFp4) return launch_tc_proj_fp4(a, stream, pdl);
    switch (a.p.TP) {
        case 16: return bits == 4 ? tc_launch<4, 16>(a, stream, pdl) : tc_launch<5, 16>(a, stream, pdl);
        case 32: return bits == 4 ? tc_launch<4, 32>(a, stream, pdl) : tc_launch<5, 32>(a, stream, pdl);
        default: return bits == 4 ? tc_launch<4, 64>(a, stream, pdl) : tc_launch<5, 64>(a, stream, pdl);
    }
}

}  // namespace nq
