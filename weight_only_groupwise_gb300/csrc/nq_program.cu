// nq_program.cu -- recorded programs (include/nq.h, "recorded programs"): a sequence of
// projection calls, a decoder layer or a stack of layers, captured once into a CUDA graph and
// replayed with one graph launch. The pages run decode through CUDA graphs built once at
// start-up ("ninfer-ext" README, section "推荐设置"; NInfer digest, section "项目定位";
// "NInfer-4090" post, section "快速启动"); this is that step for this library's calls.
//
// Recording only checks and stores the arguments (host-side, no CUDA call). Building reserves
// the device workspace of every recorded call (so that nothing allocates while the stream is
// captured), then makes the recorded calls, in order, on a stream the program owns while that
// stream is being captured: the graph holds exactly the launches the eager calls would make,
// with their plans, tensor maps and workspace addresses. A workspace that moves later (the
// library's epoch counter changed) makes the next launch build again.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>
#include <vector>

#include "nq.h"
#include "nq_launch.h"

namespace {

enum class CallKind { kGemm, kGemmFp4, kSwiglu, kSwigluFp4, kGrouped };

struct RecordedCall {
    CallKind kind;
    int bits = 0, T = 0, K = 0, N = 0;
    const void* X = nullptr;
    const void* W0 = nullptr;
    const void* S0 = nullptr;
    const void* W1 = nullptr;
    const void* S1 = nullptr;
    void* Y = nullptr;
    float gscale = 1.f, gscale1 = 1.f;  // NVFP4 tensor scales (SwiGLU: gate, up)
    std::vector<nq_group> groups;
};

}  // namespace

struct nq_program {
    std::vector<RecordedCall> calls;
    cudaStream_t capture = nullptr;   // owned; only ever captured, never runs work
    cudaGraphExec_t exec = nullptr;   // nullptr after a build with no launches
    int device = -1;                  // device of the last successful build
    unsigned long long epoch = 0;     // workspace epoch the graph was built under
    bool built = false;
    int64_t kernels = 0, builds = 0, failed = -1;
};

namespace {

void drop_graph(nq_program* p) {
    if (p->exec) cudaGraphExecDestroy(p->exec);  // a launch in flight completes first
    p->exec = nullptr;
    p->built = false;
    p->kernels = 0;
}

nq_status append(nq_program* p, RecordedCall&& c) {
    try {
        p->calls.push_back(std::move(c));
    } catch (const std::bad_alloc&) {
        return NQ_ERR_CUDA;
    }
    p->built = false;  // the graph no longer holds every recorded call
    return NQ_OK;
}

nq_status reserve_call(const RecordedCall& c) {
    switch (c.kind) {
        case CallKind::kGemm: return nq::reserve_projection_workspace(c.bits, false, c.T, c.K, c.N);
        case CallKind::kGemmFp4: return nq::reserve_projection_workspace(nq::kFp4, false, c.T, c.K, c.N);
        case CallKind::kSwiglu: return nq::reserve_projection_workspace(c.bits, true, c.T, c.K, c.N);
        case CallKind::kSwigluFp4: return nq::reserve_projection_workspace(nq::kFp4, true, c.T, c.K, c.N);
        case CallKind::kGrouped:
            return nq::reserve_grouped_workspace(c.bits, c.groups.data(), (int)c.groups.size(), c.T, c.K);
    }
    return NQ_ERR_SHAPE;
}

nq_status make_call(const RecordedCall& c, cudaStream_t s) {
    void* st = reinterpret_cast<void*>(s);
    switch (c.kind) {
        case CallKind::kGemm:
            return c.bits == 4 ? nq_gemm_q4(c.X, c.W0, c.S0, c.Y, c.T, c.K, c.N, st)
                               : nq_gemm_q5(c.X, c.W0, c.S0, c.Y, c.T, c.K, c.N, st);
        case CallKind::kGemmFp4: return nq_gemm_fp4(c.X, c.W0, c.S0, c.gscale, c.Y, c.T, c.K, c.N, st);
        case CallKind::kSwiglu:
            return c.bits == 4 ? nq_swiglu_q4(c.X, c.W0, c.S0, c.W1, c.S1, c.Y, c.T, c.K, c.N, st)
                               : nq_swiglu_q5(c.X, c.W0, c.S0, c.W1, c.S1, c.Y, c.T, c.K, c.N, st);
        case CallKind::kSwigluFp4:
            return nq_swiglu_fp4(c.X, c.W0, c.S0, c.gscale, c.W1, c.S1, c.gscale1, c.Y, c.T, c.K, c.N, st);
        case CallKind::kGrouped:
            return c.bits == 4 ? nq_gemm_q4_grouped(c.X, c.groups.data(), (int)c.groups.size(), c.T, c.K, st)
                               : nq_gemm_q5_grouped(c.X, c.groups.data(), (int)c.groups.size(), c.T, c.K, st);
    }
    return NQ_ERR_SHAPE;
}

// Kernel launches held by a captured graph (its kernel nodes).
nq_status count_kernels(cudaGraph_t g, int64_t* n_kernels) {
    size_t n = 0;
    if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess) return NQ_ERR_CUDA;
    std::vector<cudaGraphNode_t> nodes;
    try {
        nodes.resize(n);
    } catch (const std::bad_alloc&) {
        return NQ_ERR_CUDA;
    }
    if (n > 0 && cudaGraphGetNodes(g, nodes.data(), &n) != cudaSuccess) return NQ_ERR_CUDA;
    int64_t k = 0;
    for (size_t i = 0; i < n; ++i) {
        cudaGraphNodeType t;
        if (cudaGraphNodeGetType(nodes[i], &t) != cudaSuccess) return NQ_ERR_CUDA;
        if (t == cudaGraphNodeTypeKernel) ++k;
    }
    *n_kernels = k;
    return NQ_OK;
}

nq_status build(nq_program* p) {
    drop_graph(p);
    p->failed = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NQ_ERR_CUDA;
    // 1. every call's workspace, before the capture (allocation synchronises the device)
    for (size_t i = 0; i < p->calls.size(); ++i) {
        const nq_status st = reserve_call(p->calls[i]);
        if (st != NQ_OK) {
            p->failed = (int64_t)i;
            return st;
        }
    }
    const unsigned long long epoch = nq::workspace_epoch();
    // 2. capture the calls in order on the program's stream
    if (p->capture && p->device != dev) {
        cudaStreamDestroy(p->capture);
        p->capture = nullptr;
    }
    if (!p->capture && cudaStreamCreateWithFlags(&p->capture, cudaStreamNonBlocking) != cudaSuccess) {
        p->capture = nullptr;
        return NQ_ERR_CUDA;
    }
    p->device = dev;
    if (cudaStreamBeginCapture(p->capture, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return NQ_ERR_CUDA;
    nq_status st = NQ_OK;
    for (size_t i = 0; i < p->calls.size() && st == NQ_OK; ++i) {
        st = make_call(p->calls[i], p->capture);
        if (st != NQ_OK) p->failed = (int64_t)i;
    }
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(p->capture, &graph);
    if (st != NQ_OK || ec != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();  // the failed capture's error is reported here, not left pending
        return st != NQ_OK ? st : NQ_ERR_CUDA;
    }
    // 3. instantiate (a graph without nodes is kept as "nothing to launch")
    int64_t kernels = 0;
    size_t nodes = 0;
    st = count_kernels(graph, &kernels);
    if (st == NQ_OK && cudaGraphGetNodes(graph, nullptr, &nodes) != cudaSuccess) st = NQ_ERR_CUDA;
    cudaGraphExec_t exec = nullptr;
    if (st == NQ_OK && nodes > 0 && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
        cudaGetLastError();
        exec = nullptr;
        st = NQ_ERR_CUDA;
    }
    cudaGraphDestroy(graph);
    if (st != NQ_OK) return st;
    p->exec = exec;
    p->kernels = kernels;
    p->epoch = epoch;
    p->built = true;
    ++p->builds;
    return NQ_OK;
}

}  // namespace

extern "C" {

nq_status nq_program_create(nq_program** out) {
    if (!out) return NQ_ERR_NULL;
    *out = new (std::nothrow) nq_program();
    return *out ? NQ_OK : NQ_ERR_CUDA;
}

nq_status nq_program_gemm(nq_program* prog, int bits, const void* X, const void* Wq, const void* S, void* Y, int T,
                          int K, int N) {
    if (!prog) return NQ_ERR_NULL;
    if (bits != 4 && bits != 5) return NQ_ERR_SHAPE;
    const nq_status st = nq::check_projection_args(bits, false, X, Wq, S, nullptr, nullptr, Y, T, K, N);
    if (st != NQ_OK || T == 0 || N == 0) return st;
    RecordedCall c;
    c.kind = CallKind::kGemm;
    c.bits = bits;
    c.T = T;
    c.K = K;
    c.N = N;
    c.X = X;
    c.W0 = Wq;
    c.S0 = S;
    c.Y = Y;
    return append(prog, std::move(c));
}

nq_status nq_program_gemm_fp4(nq_program* prog, const void* X, const void* Wq, const void* S, float global_scale,
                              void* Y, int T, int K, int N) {
    if (!prog) return NQ_ERR_NULL;
    const nq_status st = nq::check_projection_args(nq::kFp4, false, X, Wq, S, nullptr, nullptr, Y, T, K, N);
    if (st != NQ_OK || T == 0 || N == 0) return st;
    RecordedCall c;
    c.kind = CallKind::kGemmFp4;
    c.bits = nq::kFp4;
    c.T = T;
    c.K = K;
    c.N = N;
    c.X = X;
    c.W0 = Wq;
    c.S0 = S;
    c.Y = Y;
    c.gscale = global_scale;
    return append(prog, std::move(c));
}

nq_status nq_program_swiglu(nq_program* prog, int bits, const void* X, const void* Wg, const void* Sg,
                            const void* Wu, const void* Su, void* H, int T, int K, int N) {
    if (!prog) return NQ_ERR_NULL;
    if (bits != 4 && bits != 5) return NQ_ERR_SHAPE;
    const nq_status st = nq::check_projection_args(bits, true, X, Wg, Sg, Wu, Su, H, T, K, N);
    if (st != NQ_OK || T == 0 || N == 0) return st;
    RecordedCall c;
    c.kind = CallKind::kSwiglu;
    c.bits = bits;
    c.T = T;
    c.K = K;
    c.N = N;
    c.X = X;
    c.W0 = Wg;
    c.S0 = Sg;
    c.W1 = Wu;
    c.S1 = Su;
    c.Y = H;
    return append(prog, std::move(c));
}

nq_status nq_program_swiglu_fp4(nq_program* prog, const void* X, const void* Wg, const void* Sg, float gate_scale,
                                const void* Wu, const void* Su, float up_scale, void* H, int T, int K, int N) {
    if (!prog) return NQ_ERR_NULL;
    const nq_status st = nq::check_projection_args(nq::kFp4, true, X, Wg, Sg, Wu, Su, H, T, K, N);
    if (st != NQ_OK || T == 0 || N == 0) return st;
    RecordedCall c;
    c.kind = CallKind::kSwigluFp4;
    c.bits = nq::kFp4;
    c.T = T;
    c.K = K;
    c.N = N;
    c.X = X;
    c.W0 = Wg;
    c.S0 = Sg;
    c.W1 = Wu;
    c.S1 = Su;
    c.Y = H;
    c.gscale = gate_scale;
    c.gscale1 = up_scale;
    return append(prog, std::move(c));
}

nq_status nq_program_grouped(nq_program* prog, int bits, const void* X, const nq_group* groups, int count, int T,
                             int K) {
    if (!prog) return NQ_ERR_NULL;
    if (bits != 4 && bits != 5) return NQ_ERR_SHAPE;
    const nq_status st = nq::check_grouped_args(bits, X, groups, count, T, K);
    if (st != NQ_OK || T == 0) return st;
    RecordedCall c;
    c.kind = CallKind::kGrouped;
    c.bits = bits;
    c.T = T;
    c.K = K;
    c.X = X;
    try {
        c.groups.assign(groups, groups + count);
    } catch (const std::bad_alloc&) {
        return NQ_ERR_CUDA;
    }
    return append(prog, std::move(c));
}

nq_status nq_program_build(nq_program* prog) {
    if (!prog) return NQ_ERR_NULL;
    return build(prog);
}

nq_status nq_program_launch(nq_program* prog, void* stream) {
    if (!prog) return NQ_ERR_NULL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NQ_ERR_CUDA;
    if (prog->built && prog->device != dev) return NQ_ERR_DEVICE;
    if (!prog->built || prog->epoch != nq::workspace_epoch()) {
        const nq_status st = build(prog);
        if (st != NQ_OK) return st;
    }
    if (!prog->exec) return NQ_OK;  // nothing recorded launches a kernel
    return cudaGraphLaunch(prog->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

nq_status nq_program_info(const nq_program* prog, int64_t out[4]) {
    if (!prog || !out) return NQ_ERR_NULL;
    out[0] = (int64_t)prog->calls.size();
    out[1] = prog->built ? prog->kernels : 0;
    out[2] = prog->builds;
    out[3] = prog->failed;
    return NQ_OK;
}

void nq_program_destroy(nq_program* prog) {
    if (!prog) return;
    drop_graph(prog);
    if (prog->capture) cudaStreamDestroy(prog->capture);
    delete prog;
}

}  // extern "C"
