// nq_launch.h -- internal launchers of the projection kernel instantiations.
#pragma once

#include <cuda_runtime.h>

#include "nq_proj.cuh"
#include "nq_tc.cuh"

struct nq_group;

namespace nq {

// Large-batch tensor-core kernel (nq_tc.cuh): the activation tensor map (false if the driver
// entry point is missing or rejects the view) and the launch.
bool encode_x_map(CUtensorMap* map, const void* X, int T, int K, int TP);
// Looks up the driver's tensor-map encoder once (later calls reuse it); false if it is
// missing. Recorded programs call it before a stream capture, where the lookup may not run.
bool tensor_maps_available();
bool encode_weight_maps(CUtensorMap* wmap, CUtensorMap* smap, const void* W, const void* S, int bits, int K, int N,
                        int TP);
cudaError_t launch_tc_proj(int bits, const TcArgs& a, cudaStream_t stream, bool pdl);
cudaError_t launch_tc_proj_fp4(const TcArgs& a, cudaStream_t stream, bool pdl);
// The two launches of a SwiGLU block (mode kTcOutGate, then kTcOutSwiglu), 4- or 5-bit codes
// or NVFP4 weights (bits 14).
cudaError_t launch_tc_proj_swiglu(int bits, int mode, const TcArgs& a, cudaStream_t stream, bool pdl);

// Bound of every device-side wait for later launches (nq_wait_limit; NQ_WAIT_NS).
unsigned long long wait_limit_ns();

// Host-side argument checks of the projection and grouped calls (an nq_status; NQ_OK for an
// empty problem), the reservation of the workspace a call of that shape will use (nothing is
// launched), and the workspace epoch, bumped whenever a device workspace buffer is allocated,
// moved or freed. Recorded programs (nq_program.cu) are built on these.
int check_projection_args(int bits, bool swiglu, const void* X, const void* W0, const void* S0, const void* W1,
                          const void* S1, const void* Y, int T, int K, int N);
int check_grouped_args(int bits, const void* X, const nq_group* groups, int count, int T, int K);
int reserve_projection_workspace(int bits, bool swiglu, int T, int K, int N);
int reserve_grouped_workspace(int bits, const nq_group* groups, int count, int T, int K);
unsigned long long workspace_epoch();

// Reports and clears the error word of nq_gemm_q4_noalloc's fixed scratch on device `dev`
// (NQ_OK if that device never ran it). The caller has synchronised the device.
int noalloc_take_error(int dev);

// Launch proj_kernel<BITS, SWIGLU> with a.p's grid and shared memory on `stream`.
// pdl: allow programmatic dependent launch behind the preceding kernel of the stream.
cudaError_t launch_proj_q4(const ProjArgs& a, cudaStream_t stream, bool pdl);
cudaError_t launch_proj_q5(const ProjArgs& a, cudaStream_t stream, bool pdl);
cudaError_t launch_proj_swiglu_q4(const ProjArgs& a, cudaStream_t stream, bool pdl);
cudaError_t launch_proj_swiglu_q5(const ProjArgs& a, cudaStream_t stream, bool pdl);
cudaError_t launch_proj_fp4(const ProjArgs& a, cudaStream_t stream, bool pdl);
cudaError_t launch_proj_swiglu_fp4(const ProjArgs& a, cudaStream_t stream, bool pdl);

// Slab clusters of S blocks that can be resident at once for the slab-cluster
// instantiation with `smem` bytes of shared memory per block (cudaOccupancyMaxActiveClusters);
// 0 if none.
int cluster_capacity_q4(int S, int smem);
int cluster_capacity_q5(int S, int smem);
int cluster_capacity_swiglu_q4(int S, int smem);
int cluster_capacity_swiglu_q5(int S, int smem);

template <int BITS, bool SWIGLU, bool F16, int EVEN, bool CLU>
cudaError_t launch_proj_t(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    auto kern = proj_kernel<BITS, SWIGLU, F16, EVEN, CLU>;
    // The shared-memory opt-in is per device; set it on every launch of a new size class
    // (cheap: the driver caches it) rather than tracking devices here.
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
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = a.p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    // A slab-cluster launch behind another projection kernel started late with dependent
    // launch allowed (measured: +10 us per SwiGLU block); it goes without.
    attr[0].val.programmaticStreamSerializationAllowed = (pdl && !CLU) ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (CLU) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = a.p.cl;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int BITS, bool SWIGLU>
int cluster_capacity_t(int S, int smem) {
    auto kern = proj_kernel<BITS, SWIGLU, false, 0, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// The operand type is part of the plan (a.p.f16): fp16 operands for small T, bf16 otherwise.
// Up to four tokens sit in the even MMA columns (EVEN = 1, 2 for fp16; 4 for bf16 with
// T = 3, 4): the tile epilogue then scales half the accumulators. Slab clusters (a.p.cl > 1,
// bf16 only) have their own instantiation.
static_assert(NQ_F16_MAX_T <= 2, "fp16-operand batches fit the two-token even layout");

template <int BITS, bool SWIGLU>
cudaError_t launch_proj(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    if (a.p.cl > 1) return launch_proj_t<BITS, SWIGLU, false, 0, true>(a, stream, pdl);
    if (!a.p.f16)
        return a.p.T <= 4 ? launch_proj_t<BITS, SWIGLU, false, 4, false>(a, stream, pdl)
                          : launch_proj_t<BITS, SWIGLU, false, 0, false>(a, stream, pdl);
    return a.p.T == 1 ? launch_proj_t<BITS, SWIGLU, true, 1, false>(a, stream, pdl)
                      : launch_proj_t<BITS, SWIGLU, true, 2, false>(a, stream, pdl);
}

// NVFP4 weights decode to fp16 at every T: only the fp16-operand instantiations exist, with
// up to 1, 2 or 4 tokens in the even columns, or up to eight in columns 0..7.
template <int BITS, bool SWIGLU = false>
cudaError_t launch_proj_f16_only(const ProjArgs& a, cudaStream_t stream, bool pdl) {
    if (a.p.T == 1) return launch_proj_t<BITS, SWIGLU, true, 1, false>(a, stream, pdl);
    if (a.p.T == 2) return launch_proj_t<BITS, SWIGLU, true, 2, false>(a, stream, pdl);
    return a.p.T <= 4 ? launch_proj_t<BITS, SWIGLU, true, 4, false>(a, stream, pdl)
                      : launch_proj_t<BITS, SWIGLU, true, 0, false>(a, stream, pdl);
}

}  // namespace nq
