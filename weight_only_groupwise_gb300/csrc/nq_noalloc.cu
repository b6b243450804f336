// nq_noalloc.cu -- nq_gemm_q4_noalloc: the Q4 projection for callers that cannot allocate
// device memory.
//
// nq_gemm_q4 keeps its split-K scratch (partial sums, tickets, an error word) in a workspace
// that the library allocates with cudaMalloc on first use. Some callers cannot let that
// happen: plug-ins whose host framework owns all device memory and forbids allocations
// after start-up, and processes on a fixed memory budget where a late allocation could fail
// (or synchronise the device) in the middle of serving. This entry point runs the
// same kernel with its scratch in a fixed-size array that exists in device memory for as
// long as the library is loaded, so it never calls cudaMalloc, cudaFree or any allocating
// routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "nq.h"
#include "nq_launch.h"

using namespace nq;

namespace {

// Scratch limits of this entry point: up to kStaticSlots partial-sum slots (1 KB each) and
// kStaticTickets split-K tickets, about 2.1 MB in all. Every GPU that loads the library
// holds this array until the process exits.
constexpr long long kStaticSlots = 2048;
constexpr long long kStaticTickets = 4096;
constexpr size_t kStaticTicketOff = 256;                         // after the error word
constexpr size_t kStaticPartialOff = kStaticTicketOff + kStaticTickets * 4;
constexpr size_t kStaticBytes = kStaticPartialOff + kStaticSlots * kPartialFloats * sizeof(float);

// The scratch itself. In host code this name is only a stand-in for the symbol, not a
// device address: the host looks its address up with cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch[kMaxDev] = {};   // device address of g_static_scratch, per device
int g_sms[kMaxDev] = {};

bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Once per device, with that device current: check it is an sm_103 GPU and look up the
// device address of the scratch array. Returns a status; *scratch and *sms on success.
nq_status device_setup(void** scratch, int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDev) return NQ_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch[dev]) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return NQ_ERR_CUDA;
        if (major != 10 || minor != 3) return NQ_ERR_DEVICE;
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return NQ_ERR_CUDA;
        g_scratch[dev] = ptr;
        g_sms[dev] = n;
    }
    *scratch = g_scratch[dev];
    *sms = g_sms[dev];
    return NQ_OK;
}

}  // namespace

namespace nq {
// The error word of the fixed scratch on device `dev`: a bounded wait that ran out inside an
// nq_gemm_q4_noalloc kernel set it. Reported and cleared here (with the tickets, which an
// aborted call may have left part-counted) for nq_device_error; the caller has synchronised.
int noalloc_take_error(int dev) {
    if (dev < 0 || dev >= kMaxDev) return NQ_OK;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        scratch = g_scratch[dev];
    }
    if (!scratch) return NQ_OK;
    int err = 0;
    if (cudaMemcpy(&err, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NQ_ERR_CUDA;
    if (err == 0) return NQ_OK;
    if (cudaMemset(scratch, 0, kStaticPartialOff) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        return NQ_ERR_CUDA;
    return NQ_ERR_TIMEOUT;
}
}  // namespace nq

extern "C" nq_status nq_gemm_q4_noalloc(const void* X, const void* Wq, const void* S, void* Y, int T, int K, int N,
                                        void* stream) {
    if (T < 0 || T > kMaxT || K < 0 || N < 0 || K > (1 << 20) || N > (1 << 20) || K % kGroup || N % kTileRows)
        return NQ_ERR_SHAPE;
    if (T == 0 || N == 0) return NQ_OK;
    if (!X || !Wq || !S || !Y) return NQ_ERR_NULL;
    if (misaligned16(X) || misaligned16(Wq) || misaligned16(S) || misaligned16(Y)) return NQ_ERR_ALIGN;
    const size_t xb = (size_t)T * K * 2, yb = (size_t)T * N * 2;
    const size_t wb = (size_t)K * N / 2, sb = (size_t)N * (K / kGroup) * 2;
    if (overlaps(Y, yb, X, xb) || overlaps(Y, yb, Wq, wb) || overlaps(Y, yb, S, sb)) return NQ_ERR_ALIAS;
    void* scratch = nullptr;
    int sms = 0;
    nq_status st = device_setup(&scratch, &sms);
    if (st != NQ_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) return cudaMemsetAsync(Y, 0, yb, s) == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
    // Batches above kSliceT tokens run as one launch per slice (as nq_gemm_q4). Both slice
    // sizes (full slices and the remainder) are planned and checked before anything runs.
    const int full = T < kSliceT ? T : kSliceT, rest = T > kSliceT ? T % kSliceT : 0;
    Plan plans[2];
    for (int i = 0; i < 2; ++i) {
        const int tn = i == 0 ? full : rest;
        if (tn == 0) continue;
        if (!make_plan(4, 0, tn, K, N, sms, plans[i])) return NQ_ERR_SHAPE;
        if (plans[i].slots > kStaticSlots || plans[i].RP > kStaticTickets) return NQ_ERR_SCRATCH;
    }
    uint8_t* base = static_cast<uint8_t*>(scratch);
    for (int t0 = 0; t0 < T; t0 += kSliceT) {
        ProjArgs a;
        a.p = T - t0 >= kSliceT || rest == 0 ? plans[0] : plans[1];
        a.q = a.p;  // stream-K only (no slab clusters)
        // The array keeps the previous call's contents: this launch's tickets must start at
        // zero, so clear them on the call's stream (no allocation involved). The error word is
        // left alone: it stays set until nq_device_error reports it.
        if (cudaMemsetAsync(base + kStaticTicketOff, 0, (size_t)a.p.RP * 4, s) != cudaSuccess) return NQ_ERR_CUDA;
        a.X = static_cast<const uint16_t*>(X) + (size_t)t0 * K;
        a.W0 = static_cast<const uint8_t*>(Wq);
        a.W1 = static_cast<const uint8_t*>(Wq);
        a.S0 = static_cast<const uint8_t*>(S);
        a.S1 = static_cast<const uint8_t*>(S);
        a.Y = static_cast<uint16_t*>(Y) + (size_t)t0 * N;
        a.dev_err = reinterpret_cast<int*>(base);
        a.tickets = reinterpret_cast<int*>(base + kStaticTicketOff);
        a.partials = reinterpret_cast<float*>(base + kStaticPartialOff);
        a.wait_ns = wait_limit_ns();
        if (launch_proj_q4(a, s, false) != cudaSuccess) return NQ_ERR_CUDA;
    }
    return NQ_OK;
}
