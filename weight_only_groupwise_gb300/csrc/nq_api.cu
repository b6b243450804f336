// nq_api.cu -- the C ABI of include/nq.h: argument checks, the per-device workspace, the
// offline repack kernels, the debug dequantisation kernels and the projection launches.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "nq.h"
#include "nq_launch.h"

using namespace nq;

namespace {

// ---------------------------------------------------------------- repack kernels

// Canonical -> packed codes. One thread per (tile, lane): gathers the lane's 32 codes of the
// tile from the canonical [N][K/8] nibble words (and [N][K/32] high words for Q5) and writes
// its four fragment words (+ one high word). Nibble slot i of fragment word j of lane l holds
// the code at row l/4 + 8*((i&3)>>1), column 16j + 2(l%4) + 8*(i&1) + (i>>2) of the tile; its
// high bit (Q5) goes to bit j + 4*(i&3) + 16*(i>>2) of the lane's high word. This is the
// order decode_q4 / decode_q5 turn into m16n8k16 A fragments.
template <int BITS>
__global__ void pack_codes_kernel(const uint32_t* __restrict__ wn, const uint32_t* __restrict__ wh,
                                  int K, int N, uint8_t* __restrict__ out) {
    const int G = K / kGroup;
    const long long total = (long long)(N / kTileRows) * G * 32;
    constexpr int TB = BITS == 4 ? kQ4TileBytes : kQ5TileBytes;
    const int kw8 = K / 8, kw32 = K / 32;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int lane = (int)(idx & 31);
        const long long tile = idx >> 5;
        const int rt = (int)(tile / G), g = (int)(tile % G);
        const int gid = lane >> 2, c = lane & 3;
        uint32_t words[4];
        uint32_t hw = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t wv = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int sm = i & 3, hi = i >> 2;
                const int row = gid + 8 * (sm >> 1);
                const int k = g * kGroup + 16 * j + 2 * c + 8 * (sm & 1) + hi;
                const int n = rt * kTileRows + row;
                const uint32_t nib = (wn[(size_t)n * kw8 + (k >> 3)] >> (4 * (k & 7))) & 0xFu;
                wv |= nib << (4 * i);
                if (BITS == 5) {
                    const uint32_t bit = (wh[(size_t)n * kw32 + (k >> 5)] >> (k & 31)) & 1u;
                    hw |= bit << (j + 4 * sm + 16 * hi);
                }
            }
            words[j] = wv;
        }
        uint8_t* base = out + packed_code_off(rt, g, G, TB);  // codes buffer
        reinterpret_cast<uint4*>(base)[lane] = make_uint4(words[0], words[1], words[2], words[3]);
        if (BITS == 5) reinterpret_cast<uint32_t*>(base + 512)[lane] = hw;
    }
}

// Canonical [N][K/64] fp16 scales -> the packed scale buffer: per tile 16 halves ordered
// (r, r+8) for r = 0..7.
__global__ void pack_scales_kernel(const uint16_t* __restrict__ s, int K, int N, uint8_t* __restrict__ out) {
    const int G = K / kGroup;
    const long long total = (long long)(N / kTileRows) * G * 16;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int e = (int)(idx & 15);
        const long long tile = idx >> 4;
        const int rt = (int)(tile / G), g = (int)(tile % G);
        const int row = (e >> 1) + 8 * (e & 1);
        reinterpret_cast<uint16_t*>(out + packed_scale_off(rt, g, G, kScaleTileBytes))[e] =
            s[(size_t)(rt * kTileRows + row) * G + g];
    }
}

// Canonical NVFP4 codes [N][K/8] (nibble i of word j = element 8j+i) -> packed code tiles:
// lane l's word j holds its registers 0..3 of K step j in bytes 0..3, register m = (row
// l/4 + 8 (m & 1), K pair 2(l%4) + 8 (m >> 1)), the even element in the low nibble.
__global__ void pack_fp4_codes_kernel(const uint32_t* __restrict__ wn, int K, int N, uint8_t* __restrict__ out) {
    const int G = K / kGroup;
    const long long total = (long long)(N / kTileRows) * G * 32;
    const int kw8 = K / 8;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int lane = (int)(idx & 31);
        const long long tile = idx >> 5;
        const int rt = (int)(tile / G), g = (int)(tile % G);
        const int gid = lane >> 2, c = lane & 3;
        uint32_t words[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t wv = 0;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int n = rt * kTileRows + gid + 8 * (m & 1);
                const int k0 = g * kGroup + 16 * j + 2 * c + 8 * (m >> 1);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = k0 + e;
                    const uint32_t code = (wn[(size_t)n * kw8 + (k >> 3)] >> (4 * (k & 7))) & 0xFu;
                    wv |= code << (8 * m + 4 * e);
                }
            }
            words[j] = wv;
        }
        reinterpret_cast<uint4*>(out + packed_code_off(rt, g, G, kQ4TileBytes))[lane] =
            make_uint4(words[0], words[1], words[2], words[3]);
    }
}

// Canonical e4m3 block scales [N][K/16] -> packed scale tiles: byte 8 r + 2 j + h of tile (rt, g)
// is the scale of row 16 rt + r + 8 h, K step j of group g.
__global__ void pack_fp4_scales_kernel(const uint8_t* __restrict__ sf, int K, int N, uint8_t* __restrict__ out) {
    const int G = K / kGroup;
    const long long total = (long long)(N / kTileRows) * G * kFp4ScaleTileBytes;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(idx % kFp4ScaleTileBytes);
        const long long tile = idx / kFp4ScaleTileBytes;
        const int rt = (int)(tile / G), g = (int)(tile % G);
        const int r = b >> 3, j = (b >> 1) & 3, h = b & 1;
        out[packed_scale_off(rt, g, G, kFp4ScaleTileBytes) + b] =
            sf[(size_t)(rt * kTileRows + r + 8 * h) * (K / 16) + g * 4 + j];
    }
}

// Packed NVFP4 pair -> fp32 W[n][k] = g * (fp16 register value), through decode_fp4, the
// projection kernel's own decoder (the register value is exactly scale * element).
__global__ void dequant_fp4_kernel(const uint8_t* __restrict__ wq, const uint8_t* __restrict__ sq, float gs, int K,
                                   int N, float* __restrict__ w) {
    const int G = K / kGroup;
    const long long total = (long long)(N / kTileRows) * G * 32;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int lane = (int)(idx & 31);
        const long long tile = idx >> 5;
        const int rt = (int)(tile / G), g = (int)(tile % G);
        const int gid = lane >> 2, c = lane & 3;
        const uint4 wv = reinterpret_cast<const uint4*>(wq + packed_code_off(rt, g, G, kQ4TileBytes))[lane];
        const uint2 sc = *reinterpret_cast<const uint2*>(sq + packed_scale_off(rt, g, G, kFp4ScaleTileBytes) + gid * 8);
        const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
        const uint32_t ss[4] = {sc.x, sc.x >> 16, sc.y, sc.y >> 16};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t a[4];
            decode_fp4(ws[j], ss[j], a);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int row = gid + 8 * (m & 1);
                const int k = g * kGroup + 16 * j + 2 * c + 8 * (m >> 1);
                float* dst = w + (size_t)(rt * kTileRows + row) * K + k;
                dst[0] = gs * __half2float(__ushort_as_half((unsigned short)(a[m] & 0xFFFFu)));
                dst[1] = gs * __half2float(__ushort_as_half((unsigned short)(a[m] >> 16)));
            }
        }
    }
}

// Packed -> fp32 W[n][k], decoding with the projection kernels' own decoders:
//   F16 (the T <= 2 kernels): decode_q4 / decode_q5<J>, a lower-K half holds 1024 + q and an
//     upper-K half 1024 + 16 q (fp16);
//   bf16 (the T >= 3 kernels): decode_q4_bf16 / decode_q5_bf16<J>, every half holds 128 + q.
// Then w = (float)s * (q - z); every step is exact in fp32.
template <int BITS, int J, bool F16>
__device__ __forceinline__ void decode_for_dump(uint32_t w, uint32_t h, uint32_t a[4]) {
    if constexpr (F16) {
        if constexpr (BITS == 4) decode_q4(w, a); else decode_q5<J>(w, h, a);
    } else {
        if constexpr (BITS == 4) decode_q4_bf16(w, a); else decode_q5_bf16<J>(w, h, a);
    }
}

template <int BITS, bool F16, int J>
__device__ __forceinline__ void dump_step(uint32_t w, uint32_t hb, int rt, int g, int gid, int c, int K, float s_lo,
                                          float s_hi, float* __restrict__ out) {
    constexpr float z = BITS == 4 ? 8.0f : 16.0f;
    uint32_t a[4];
    decode_for_dump<BITS, J, F16>(w, hb, a);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        // register m: rows r (m even) / r+8 (m odd), K pair k (m < 2) / k+8 (m >= 2)
        const int row = gid + 8 * (m & 1);
        const int k = g * kGroup + 16 * J + 2 * c + 8 * (m >> 1);
        const float s = (m & 1) ? s_hi : s_lo;
        float v0, v1;
        if constexpr (F16) {
            const float step = m < 2 ? 1.0f : 16.0f;
            v0 = (__half2float(__ushort_as_half((unsigned short)(a[m] & 0xFFFFu))) - 1024.0f) / step;
            v1 = (__half2float(__ushort_as_half((unsigned short)(a[m] >> 16))) - 1024.0f) / step;
        } else {
            v0 = __bfloat162float(__ushort_as_bfloat16((unsigned short)(a[m] & 0xFFFFu))) - 128.0f;
            v1 = __bfloat162float(__ushort_as_bfloat16((unsigned short)(a[m] >> 16))) - 128.0f;
        }
        float* dst = out + (size_t)(rt * kTileRows + row) * K + k;
        dst[0] = s * (v0 - z);
        dst[1] = s * (v1 - z);
    }
}

template <int BITS, bool F16>
__global__ void dequant_kernel(const uint8_t* __restrict__ wq, const uint8_t* __restrict__ sq, int K, int N,
                               float* __restrict__ w) {
    const int G = K / kGroup;
    const long long total = (long long)(N / kTileRows) * G * 32;
    constexpr int TB = BITS == 4 ? kQ4TileBytes : kQ5TileBytes;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int lane = (int)(idx & 31);
        const long long tile = idx >> 5;
        const int rt = (int)(tile / G), g = (int)(tile % G);
        const int gid = lane >> 2, c = lane & 3;
        const uint8_t* tb = wq + packed_code_off(rt, g, G, TB);
        const uint4 wv = reinterpret_cast<const uint4*>(tb)[lane];
        const uint32_t hb = BITS == 5 ? reinterpret_cast<const uint32_t*>(tb + 512)[lane] : 0u;
        const uint16_t* st = reinterpret_cast<const uint16_t*>(sq + packed_scale_off(rt, g, G, kScaleTileBytes));
        const float s_lo = __half2float(__ushort_as_half(st[2 * gid]));
        const float s_hi = __half2float(__ushort_as_half(st[2 * gid + 1]));
        dump_step<BITS, F16, 0>(wv.x, hb, rt, g, gid, c, K, s_lo, s_hi, w);
        dump_step<BITS, F16, 1>(wv.y, hb, rt, g, gid, c, K, s_lo, s_hi, w);
        dump_step<BITS, F16, 2>(wv.z, hb, rt, g, gid, c, K, s_lo, s_hi, w);
        dump_step<BITS, F16, 3>(wv.w, hb, rt, g, gid, c, K, s_lo, s_hi, w);
    }
}

// ---------------------------------------------------------------- per-device state

struct DevState {
    bool init = false;
    int major = 0, minor = 0, sms = 0;
    uint8_t* ws = nullptr;     // [err: 256 B][tickets][partials]
    long long slots_cap = 0;
    long long tickets_cap = 0;
    // resident slab clusters per [S][bits == 5][swiglu], -1 until queried
    int cluster_cap[kMaxCluster + 1][2][2];
    // large-batch tensor-core kernel: [tickets: 4 B per row block, 256-B rounded][partials]
    uint8_t* tc_ws = nullptr;
    long long tc_tickets = 0, tc_floats = 0;
    float* tc_gate = nullptr;   // fp32 gate outputs of a tensor-core SwiGLU call, [T][N]
    long long tc_gate_floats = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevState g_dev[kMaxDevices];
bool g_pdl = true;
bool g_cluster = false;
bool g_env_read = false;
bool g_tc = true;
unsigned long long g_wait_ns = (unsigned long long)kWaitTimeoutNs;
// Bumped whenever a device workspace buffer is allocated, moved or freed: a recorded program
// built under another value holds stale workspace addresses and is built again.
std::atomic<unsigned long long> g_ws_epoch{0};

// Reads NQ_PDL, NQ_CLUSTER and NQ_WAIT_NS once (the first call that needs them). g_mu held.
void read_env_locked() {
    if (g_env_read) return;
    const char* e = std::getenv("NQ_PDL");
    if (e && e[0] == '0') g_pdl = false;
    const char* c = std::getenv("NQ_CLUSTER");
    if (c && c[0] == '1') g_cluster = true;
    const char* tcv = std::getenv("NQ_TC");
    if (tcv && tcv[0] == '0') g_tc = false;
    const char* w = std::getenv("NQ_WAIT_NS");
    if (w) {
        const long long v = std::atoll(w);
        if (v > 0) g_wait_ns = (unsigned long long)v;
    }
    g_env_read = true;
}

size_t ws_tickets_off() { return 256; }
size_t ws_partials_off(long long tickets_cap) {
    return 256 + (((size_t)tickets_cap * 4 + 255) / 256) * 256;
}

// Device state of the current device (initialised on first use). Returns a status.
nq_status current_device(DevState** out, int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return NQ_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    read_env_locked();
    DevState& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return NQ_ERR_CUDA;
        for (auto& a : d.cluster_cap)
            for (auto& b : a)
                for (int& c : b) c = -1;
        d.init = true;
    }
    if (d.major != 10 || d.minor != 3) return NQ_ERR_DEVICE;
    *out = &d;
    if (dev_out) *dev_out = dev;
    return NQ_OK;
}

// Make the workspace of d hold `slots` partial slots and `tickets` tickets. Growing it
// synchronises the device (old buffer may be in use) and zero-fills the new one.
nq_status ensure_workspace(DevState& d, long long slots, long long tickets) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (d.ws && slots <= d.slots_cap && tickets <= d.tickets_cap) return NQ_OK;
    long long sc = d.slots_cap > slots ? d.slots_cap : slots;
    long long tc = d.tickets_cap > tickets ? d.tickets_cap : tickets;
    if (sc < 1024) sc = 1024;
    if (tc < 4096) tc = 4096;
    const size_t bytes = ws_partials_off(tc) + (size_t)sc * kPartialFloats * sizeof(float);
    if (d.ws) {
        if (cudaDeviceSynchronize() != cudaSuccess) return NQ_ERR_CUDA;
        cudaFree(d.ws);
        d.ws = nullptr;
        d.slots_cap = d.tickets_cap = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return NQ_ERR_CUDA;
    if (cudaMemset(p, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(p);
        return NQ_ERR_CUDA;
    }
    d.ws = static_cast<uint8_t*>(p);
    d.slots_cap = sc;
    d.tickets_cap = tc;
    ++g_ws_epoch;
    return NQ_OK;
}

// The tensor-core kernel's scratch: tickets (zero between calls) and fp32 partial slots.
// Growing it synchronises the device.
nq_status ensure_tc_workspace(DevState& d, long long tickets, long long floats) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (d.tc_ws && tickets <= d.tc_tickets && floats <= d.tc_floats) return NQ_OK;
    long long tc = d.tc_tickets > tickets ? d.tc_tickets : tickets;
    long long fc = d.tc_floats > floats ? d.tc_floats : floats;
    if (tc < 1024) tc = 1024;
    const size_t toff = (((size_t)tc * 4 + 255) / 256) * 256;
    const size_t bytes = toff + (size_t)fc * sizeof(float);
    if (d.tc_ws) {
        if (cudaDeviceSynchronize() != cudaSuccess) return NQ_ERR_CUDA;
        cudaFree(d.tc_ws);
        d.tc_ws = nullptr;
        d.tc_tickets = d.tc_floats = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return NQ_ERR_CUDA;
    if (cudaMemset(p, 0, toff) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(p);
        return NQ_ERR_CUDA;
    }
    d.tc_ws = static_cast<uint8_t*>(p);
    d.tc_tickets = tc;
    d.tc_floats = fc;
    ++g_ws_epoch;
    return NQ_OK;
}

// The fp32 gate buffer of tensor-core SwiGLU calls, grown to at least `floats`.
nq_status ensure_tc_gate(DevState& d, long long floats) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (d.tc_gate && floats <= d.tc_gate_floats) return NQ_OK;
    if (d.tc_gate) {
        if (cudaDeviceSynchronize() != cudaSuccess) return NQ_ERR_CUDA;
        cudaFree(d.tc_gate);
        d.tc_gate = nullptr;
        d.tc_gate_floats = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, (size_t)floats * sizeof(float)) != cudaSuccess) return NQ_ERR_CUDA;
    d.tc_gate = static_cast<float*>(p);
    d.tc_gate_floats = floats;
    ++g_ws_epoch;
    return NQ_OK;
}

// ---------------------------------------------------------------- argument checks

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

constexpr long long kMaxDim = 1 << 20;  // K, N bound: keeps every index well inside 64 bits

nq_status check_shape(int K, int N) {
    if (K < 0 || N < 0 || K > kMaxDim || N > kMaxDim) return NQ_ERR_SHAPE;
    if (K % kGroup != 0 || N % kTileRows != 0) return NQ_ERR_SHAPE;
    return NQ_OK;
}

// Packed code bytes (K*N/2, or 5*K*N/8 for Q5) and packed scale bytes (N*K/32: fp16 per 64;
// NVFP4: N*K/16, e4m3 per 16).
size_t packed_bytes(int bits, int K, int N) { return (size_t)K * N / 8 * (bits == 5 ? 5 : 4); }
size_t scale_bytes(int K, int N, int bits = 4) {
    return bits == kFp4 ? (size_t)N * (K / 16) : (size_t)N * (K / kGroup) * 2;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int grid_for(long long work, int per_block) {
    long long b = (work + per_block - 1) / per_block;
    if (b > 65535LL * 16) b = 65535LL * 16;
    return (int)(b < 1 ? 1 : b);
}

// Slab clusters of S blocks to launch: as many as can be resident at once (queried once per
// device and instantiation; every plan of a slab-cluster instantiation needs more than half
// of an SM's shared memory, so one block per SM), at most one block per SM.
int resident_clusters(DevState& d, int bits, bool swiglu, int S) {
    int& c = d.cluster_cap[S][bits == 5 ? 1 : 0][swiglu ? 1 : 0];
    if (c < 0) {
        const int smem = kSmemLimit;
        if (bits == 4)
            c = swiglu ? cluster_capacity_swiglu_q4(S, smem) : cluster_capacity_q4(S, smem);
        else
            c = swiglu ? cluster_capacity_swiglu_q5(S, smem) : cluster_capacity_q5(S, smem);
    }
    const int cap = d.sms / S;
    return c < cap ? c : cap;
}

// The work split of one launch of T <= kSliceT tokens: the stream-K plan, or slab clusters when
// K needs 2..kMaxCluster slabs (bf16 operands), enough clusters fit and they are switched on.
bool choose_plans(int bits, bool swiglu, int T, int K, int N, DevState& d, Plan& p, Plan& q) {
    if (!make_plan(bits, swiglu ? 1 : 0, T, K, N, d.sms, p)) return false;
    q = p;
    if (g_cluster && p.S >= 2 && p.S <= kMaxCluster && !p.f16) {
        Plan p2, q2;
        const int C = resident_clusters(d, bits, swiglu, p.S);
        if (C > 0 && make_cluster_plans(bits, swiglu ? 1 : 0, T, K, N, C, p2, q2)) {
            p = p2;
            q = q2;
        }
    }
    return true;
}

// Shared body of the projection entry points (Q4/Q5 GEMM, Q4/Q5 SwiGLU). W0/S0: the weight
// (gemm) or the gate weight (swiglu); W1/S1: the up weight (swiglu only). T up to kSliceT runs
// as one launch; larger batches (up to kMaxT) as one launch per slice of kSliceT tokens, each
// streaming the weights again. Every slice's plan and the workspace are settled before the
// first launch, so an error still launches nothing.
// The host-side argument checks of a projection call, in order: shape, then (for a non-empty
// problem) NULL, alignment, aliasing. NQ_OK for an empty problem.
nq_status projection_args(int bits, bool swiglu, const void* X, const void* W0, const void* S0, const void* W1,
                          const void* S1, const void* Y, int T, int K, int N) {
    if (T < 0 || T > kMaxT) return NQ_ERR_SHAPE;
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    if (T == 0 || N == 0) return NQ_OK;  // empty output
    if (!X || !W0 || !S0 || !Y || (swiglu && (!W1 || !S1))) return NQ_ERR_NULL;
    if (misaligned(X) || misaligned(W0) || misaligned(S0) || misaligned(Y) ||
        (swiglu && (misaligned(W1) || misaligned(S1))))
        return NQ_ERR_ALIGN;
    const size_t xb = (size_t)T * K * 2, yb = (size_t)T * N * 2;
    const size_t wb = packed_bytes(bits, K, N), sb = scale_bytes(K, N, bits);
    if (overlap(Y, yb, X, xb) || overlap(Y, yb, W0, wb) || overlap(Y, yb, S0, sb) ||
        (swiglu && (overlap(Y, yb, W1, wb) || overlap(Y, yb, S1, sb))))
        return NQ_ERR_ALIAS;
    return NQ_OK;
}

nq_status project(int bits, bool swiglu, const void* X, const void* W0, const void* S0, const void* W1,
                  const void* S1, void* Y, int T, int K, int N, void* stream, float gscale = 1.f,
                  float gscale1 = 1.f) {
    nq_status st = projection_args(bits, swiglu, X, W0, S0, W1, S1, Y, T, K, N);
    if (st != NQ_OK) return st;
    if (T == 0 || N == 0) return NQ_OK;  // empty output
    DevState* d = nullptr;
    st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    if (K == 0) {  // empty sum
        return cudaMemsetAsync(Y, 0, (size_t)T * N * 2, as_stream(stream)) == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
    }
    // Larger batches: the tensor-core kernel, one weight pass per matrix. A SwiGLU block is two
    // launches on the same X: the gate projection writes fp32 G to a library buffer, the up
    // projection's epilogue writes H = silu(G) * U in bf16.
    if (g_tc && (bits == 4 || bits == 5 || bits == kFp4) && T > kSliceT && T <= kTcMaxT) {
        alignas(64) TcArgs ta;
        alignas(64) TcArgs tu;
        if (make_tc_plan(bits, T, K, N, d->sms, ta.p) && encode_x_map(&ta.xmap, X, T, K, ta.p.TP) &&
            encode_weight_maps(&ta.wmap, &ta.smap, W0, S0, bits, K, N, ta.p.TP) &&
            (!swiglu || encode_weight_maps(&tu.wmap, &tu.smap, W1, S1, bits, K, N, ta.p.TP))) {
            st = ensure_workspace(*d, 1, 1);
            if (st != NQ_OK) return st;
            st = ensure_tc_workspace(*d, ta.p.RB, ta.p.KS > 1 ? (long long)ta.p.P * kTcRows * ta.p.TP : 1);
            if (st != NQ_OK) return st;
            if (swiglu) {
                st = ensure_tc_gate(*d, (long long)T * N);
                if (st != NQ_OK) return st;
            }
            ta.W = static_cast<const uint8_t*>(W0);
            ta.S = static_cast<const uint8_t*>(S0);
            ta.Y = static_cast<uint16_t*>(Y);
            ta.G = d->tc_gate;
            ta.gscale = gscale;
            ta.tickets = reinterpret_cast<int*>(d->tc_ws);
            ta.partials = reinterpret_cast<float*>(d->tc_ws + (((size_t)d->tc_tickets * 4 + 255) / 256) * 256);
            ta.dev_err = reinterpret_cast<int*>(d->ws);
            ta.wait_ns = g_wait_ns;
            if (!swiglu) return launch_tc_proj(bits, ta, as_stream(stream), g_pdl) == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
            if (launch_tc_proj_swiglu(bits, kTcOutGate, ta, as_stream(stream), g_pdl) != cudaSuccess)
                return NQ_ERR_CUDA;
            const CUtensorMap wmap = tu.wmap, smap = tu.smap;
            tu = ta;
            tu.wmap = wmap;
            tu.smap = smap;
            tu.W = static_cast<const uint8_t*>(W1);
            tu.S = static_cast<const uint8_t*>(S1);
            tu.gscale = gscale1;
            return launch_tc_proj_swiglu(bits, kTcOutSwiglu, tu, as_stream(stream), g_pdl) == cudaSuccess ? NQ_OK
                                                                                                : NQ_ERR_CUDA;
        }
    }
    // At most two distinct slice sizes: full slices and the remainder.
    const int full = T < kSliceT ? T : kSliceT, rest = T > kSliceT ? T % kSliceT : 0;
    ProjArgs a_full, a_rest;
    if (!choose_plans(bits, swiglu, full, K, N, *d, a_full.p, a_full.q)) return NQ_ERR_SHAPE;
    long long slots = a_full.q.slots, tickets = a_full.q.RP;
    if (rest > 0) {
        if (!choose_plans(bits, swiglu, rest, K, N, *d, a_rest.p, a_rest.q)) return NQ_ERR_SHAPE;
        if (a_rest.q.slots > slots) slots = a_rest.q.slots;
    }
    st = ensure_workspace(*d, slots, tickets);
    if (st != NQ_OK) return st;
    for (int t0 = 0; t0 < T; t0 += kSliceT) {
        ProjArgs a = T - t0 >= kSliceT || rest == 0 ? a_full : a_rest;
        a.X = static_cast<const uint16_t*>(X) + (size_t)t0 * K;
        a.W0 = static_cast<const uint8_t*>(W0);
        a.S0 = static_cast<const uint8_t*>(S0);
        a.W1 = static_cast<const uint8_t*>(swiglu ? W1 : W0);
        a.S1 = static_cast<const uint8_t*>(swiglu ? S1 : S0);
        a.Y = static_cast<uint16_t*>(Y) + (size_t)t0 * N;
        a.dev_err = reinterpret_cast<int*>(d->ws);
        a.tickets = reinterpret_cast<int*>(d->ws + ws_tickets_off());
        a.partials = reinterpret_cast<float*>(d->ws + ws_partials_off(d->tickets_cap));
        a.wait_ns = g_wait_ns;
        a.gscale = gscale;
        a.gscale1 = swiglu ? gscale1 : gscale;
        cudaError_t e;
        if (bits == kFp4)
            e = swiglu ? launch_proj_swiglu_fp4(a, as_stream(stream), g_pdl) : launch_proj_fp4(a, as_stream(stream), g_pdl);
        else if (swiglu)
            e = bits == 4 ? launch_proj_swiglu_q4(a, as_stream(stream), g_pdl)
                          : launch_proj_swiglu_q5(a, as_stream(stream), g_pdl);
        else if (bits == 4)
            e = launch_proj_q4(a, as_stream(stream), g_pdl);
        else
            e = launch_proj_q5(a, as_stream(stream), g_pdl);
        if (e != cudaSuccess) return NQ_ERR_CUDA;
    }
    return NQ_OK;
}

// Several projections of the same X in one launch per slice (gemm only, no slab clusters):
// group g owns ceil(N_g / 32) consecutive row pairs of the work split.
// The host-side argument checks of a grouped call, in order (NQ_OK for T == 0).
nq_status grouped_args(int bits, const void* X, const nq_group* groups, int count, int T, int K) {
    if (!groups) return NQ_ERR_NULL;
    if (count < 1 || count > kMaxGroups || T < 0 || T > kMaxT) return NQ_ERR_SHAPE;
    for (int g = 0; g < count; ++g) {
        nq_status st = check_shape(K, groups[g].N);
        if (st != NQ_OK) return st;
        if (groups[g].N == 0) return NQ_ERR_SHAPE;
    }
    nq_status st = check_shape(K, 16);
    if (st != NQ_OK) return st;
    if (T == 0) return NQ_OK;
    if (!X) return NQ_ERR_NULL;
    if (misaligned(X)) return NQ_ERR_ALIGN;
    const size_t xb = (size_t)T * K * 2;
    for (int g = 0; g < count; ++g) {
        const nq_group& G = groups[g];
        if (!G.Wq || !G.S || !G.Y) return NQ_ERR_NULL;
        if (misaligned(G.Wq) || misaligned(G.S) || misaligned(G.Y)) return NQ_ERR_ALIGN;
    }
    for (int g = 0; g < count; ++g) {
        const size_t yb = (size_t)T * groups[g].N * 2;
        if (overlap(groups[g].Y, yb, X, xb)) return NQ_ERR_ALIAS;
        for (int h = 0; h < count; ++h) {
            if (overlap(groups[g].Y, yb, groups[h].Wq, packed_bytes(bits, K, groups[h].N)) ||
                overlap(groups[g].Y, yb, groups[h].S, scale_bytes(K, groups[h].N, bits)))
                return NQ_ERR_ALIAS;
            if (h != g && overlap(groups[g].Y, yb, groups[h].Y, (size_t)T * groups[h].N * 2)) return NQ_ERR_ALIAS;
        }
    }
    return NQ_OK;
}

nq_status project_grouped(int bits, const void* X, const nq_group* groups, int count, int T, int K, void* stream) {
    nq_status st = grouped_args(bits, X, groups, count, T, K);
    if (st != NQ_OK) return st;
    if (T == 0) return NQ_OK;
    DevState* d = nullptr;
    st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    if (K == 0) {  // empty sums
        for (int g = 0; g < count; ++g)
            if (cudaMemsetAsync(groups[g].Y, 0, (size_t)T * groups[g].N * 2, as_stream(stream)) != cudaSuccess)
                return NQ_ERR_CUDA;
        return NQ_OK;
    }
    // 8 < T <= 64: one tensor-core launch per matrix (each streams its weights once) instead of
    // 8-token slices of a grouped launch (each slice streams all of them again).
    if (g_tc && (bits == 4 || bits == 5) && T > kSliceT && T <= kTcMaxT) {
        for (int g = 0; g < count; ++g) {
            st = project(bits, false, X, groups[g].Wq, groups[g].S, nullptr, nullptr, groups[g].Y, T, K, groups[g].N,
                         stream);
            if (st != NQ_OK) return st;
        }
        return NQ_OK;
    }
    int gpair[kMaxGroups + 1];
    gpair[0] = 0;
    for (int g = 0; g < count; ++g) gpair[g + 1] = gpair[g] + (groups[g].N + 2 * kTileRows - 1) / (2 * kTileRows);
    const int n_pairs = gpair[count];
    if ((long long)n_pairs * 2 * kTileRows > kMaxDim) return NQ_ERR_SHAPE;
    const int full = T < kSliceT ? T : kSliceT, rest = T > kSliceT ? T % kSliceT : 0;
    Plan plans[2];
    for (int i = 0; i < 2; ++i) {
        const int tn = i == 0 ? full : rest;
        if (tn > 0 && !make_plan(bits, 0, tn, K, n_pairs * 2 * kTileRows, d->sms, plans[i])) return NQ_ERR_SHAPE;
    }
    long long slots = plans[0].slots;
    if (rest > 0 && plans[1].slots > slots) slots = plans[1].slots;
    st = ensure_workspace(*d, slots, n_pairs);
    if (st != NQ_OK) return st;
    for (int t0 = 0; t0 < T; t0 += kSliceT) {
        ProjArgs a;
        a.p = T - t0 >= kSliceT || rest == 0 ? plans[0] : plans[1];
        a.q = a.p;
        a.X = static_cast<const uint16_t*>(X) + (size_t)t0 * K;
        a.W0 = a.W1 = static_cast<const uint8_t*>(groups[0].Wq);
        a.S0 = a.S1 = static_cast<const uint8_t*>(groups[0].S);
        a.Y = static_cast<uint16_t*>(groups[0].Y);
        a.ngroups = count;
        for (int g = 0; g <= count; ++g) a.gpair[g] = gpair[g];
        for (int g = 0; g < count; ++g) {
            a.gW[g] = static_cast<const uint8_t*>(groups[g].Wq);
            a.gS[g] = static_cast<const uint8_t*>(groups[g].S);
            a.gY[g] = static_cast<uint16_t*>(groups[g].Y) + (size_t)t0 * groups[g].N;
            a.gN[g] = groups[g].N;
        }
        a.dev_err = reinterpret_cast<int*>(d->ws);
        a.tickets = reinterpret_cast<int*>(d->ws + ws_tickets_off());
        a.partials = reinterpret_cast<float*>(d->ws + ws_partials_off(d->tickets_cap));
        a.wait_ns = g_wait_ns;
        const cudaError_t e = bits == 4 ? launch_proj_q4(a, as_stream(stream), g_pdl)
                                        : launch_proj_q5(a, as_stream(stream), g_pdl);
        if (e != cudaSuccess) return NQ_ERR_CUDA;
    }
    return NQ_OK;
}

// The workspace a projection call of this shape will use, allocated now; nothing is launched.
// It draws the same plans as project(): the tensor-core plan where that branch applies, and
// the 8-token slice plans (the fallback of that branch, and the path of every other call).
nq_status reserve_projection(int bits, bool swiglu, int T, int K, int N) {
    if (T <= 0 || K <= 0 || N <= 0) return NQ_OK;  // empty problems use no workspace
    DevState* d = nullptr;
    nq_status st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    if (g_tc && (bits == 4 || bits == 5 || bits == kFp4) && T > kSliceT && T <= kTcMaxT) {
        TcPlan p;
        if (make_tc_plan(bits, T, K, N, d->sms, p) && tensor_maps_available()) {
            st = ensure_workspace(*d, 1, 1);
            if (st == NQ_OK) st = ensure_tc_workspace(*d, p.RB, p.KS > 1 ? (long long)p.P * kTcRows * p.TP : 1);
            if (st == NQ_OK && swiglu) st = ensure_tc_gate(*d, (long long)T * N);
            if (st != NQ_OK) return st;
        }
    }
    const int full = T < kSliceT ? T : kSliceT, rest = T > kSliceT ? T % kSliceT : 0;
    Plan p, q;
    if (!choose_plans(bits, swiglu, full, K, N, *d, p, q)) return NQ_ERR_SHAPE;
    long long slots = q.slots;
    const long long tickets = q.RP;
    if (rest > 0) {
        if (!choose_plans(bits, swiglu, rest, K, N, *d, p, q)) return NQ_ERR_SHAPE;
        if (q.slots > slots) slots = q.slots;
    }
    return ensure_workspace(*d, slots, tickets);
}

// As reserve_projection for a grouped call (its arguments already checked).
nq_status reserve_grouped(int bits, const nq_group* groups, int count, int T, int K) {
    if (T <= 0 || K <= 0) return NQ_OK;
    DevState* d = nullptr;
    nq_status st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    if (g_tc && (bits == 4 || bits == 5) && T > kSliceT && T <= kTcMaxT) {
        for (int g = 0; g < count; ++g) {
            st = reserve_projection(bits, false, T, K, groups[g].N);
            if (st != NQ_OK) return st;
        }
        return NQ_OK;
    }
    int n_pairs = 0;
    for (int g = 0; g < count; ++g) n_pairs += (groups[g].N + 2 * kTileRows - 1) / (2 * kTileRows);
    if ((long long)n_pairs * 2 * kTileRows > kMaxDim) return NQ_ERR_SHAPE;
    const int full = T < kSliceT ? T : kSliceT, rest = T > kSliceT ? T % kSliceT : 0;
    long long slots = 0;
    for (int i = 0; i < 2; ++i) {
        const int tn = i == 0 ? full : rest;
        Plan p;
        if (tn > 0) {
            if (!make_plan(bits, 0, tn, K, n_pairs * 2 * kTileRows, d->sms, p)) return NQ_ERR_SHAPE;
            if (p.slots > slots) slots = p.slots;
        }
    }
    return ensure_workspace(*d, slots, n_pairs);
}

nq_status pack(int bits, const uint32_t* wn, const uint32_t* wh, const uint16_t* s, int K, int N, void* wq_packed,
               void* s_packed, void* stream) {
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    if (K == 0 || N == 0) return NQ_OK;
    if (!wn || !s || !wq_packed || !s_packed || (bits == 5 && !wh)) return NQ_ERR_NULL;
    if (misaligned(wn) || misaligned(s) || misaligned(wq_packed) || misaligned(s_packed) ||
        (bits == 5 && misaligned(wh)))
        return NQ_ERR_ALIGN;
    const size_t ob = packed_bytes(bits, K, N), osb = scale_bytes(K, N);
    const size_t in_n = (size_t)N * K / 2, in_h = (size_t)N * K / 8, in_s = scale_bytes(K, N);
    const void* outs[2] = {wq_packed, s_packed};
    const size_t out_n[2] = {ob, osb};
    for (int i = 0; i < 2; ++i)
        if (overlap(outs[i], out_n[i], wn, in_n) || overlap(outs[i], out_n[i], s, in_s) ||
            (bits == 5 && overlap(outs[i], out_n[i], wh, in_h)))
            return NQ_ERR_ALIAS;
    if (overlap(wq_packed, ob, s_packed, osb)) return NQ_ERR_ALIAS;
    DevState* d = nullptr;
    st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    const long long lanes = (long long)(N / kTileRows) * (K / kGroup) * 32;
    uint8_t* out = static_cast<uint8_t*>(wq_packed);
    if (bits == 4)
        pack_codes_kernel<4><<<grid_for(lanes, 256), 256, 0, as_stream(stream)>>>(wn, nullptr, K, N, out);
    else
        pack_codes_kernel<5><<<grid_for(lanes, 256), 256, 0, as_stream(stream)>>>(wn, wh, K, N, out);
    if (cudaGetLastError() != cudaSuccess) return NQ_ERR_CUDA;
    pack_scales_kernel<<<grid_for(lanes / 2, 256), 256, 0, as_stream(stream)>>>(s, K, N,
                                                                               static_cast<uint8_t*>(s_packed));
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

nq_status dequant(int bits, bool f16, const void* wq, const void* sq, float* w, int K, int N, void* stream) {
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    if (K == 0 || N == 0) return NQ_OK;
    if (!wq || !sq || !w) return NQ_ERR_NULL;
    if (misaligned(wq) || misaligned(sq) || misaligned(w)) return NQ_ERR_ALIGN;
    if (overlap(w, (size_t)N * K * 4, wq, packed_bytes(bits, K, N)) || overlap(w, (size_t)N * K * 4, sq, scale_bytes(K, N)))
        return NQ_ERR_ALIAS;
    DevState* d = nullptr;
    st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    const long long lanes = (long long)(N / kTileRows) * (K / kGroup) * 32;
    const uint8_t* c = static_cast<const uint8_t*>(wq);
    const uint8_t* sc = static_cast<const uint8_t*>(sq);
    const int grid = grid_for(lanes, 256);
    cudaStream_t s = as_stream(stream);
    if (bits == 4 && f16) dequant_kernel<4, true><<<grid, 256, 0, s>>>(c, sc, K, N, w);
    if (bits == 4 && !f16) dequant_kernel<4, false><<<grid, 256, 0, s>>>(c, sc, K, N, w);
    if (bits == 5 && f16) dequant_kernel<5, true><<<grid, 256, 0, s>>>(c, sc, K, N, w);
    if (bits == 5 && !f16) dequant_kernel<5, false><<<grid, 256, 0, s>>>(c, sc, K, N, w);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

nq_status pack_fp4(const uint32_t* codes, const uint8_t* sf, int K, int N, void* wq_packed, void* s_packed,
                   void* stream) {
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    if (K == 0 || N == 0) return NQ_OK;
    if (!codes || !sf || !wq_packed || !s_packed) return NQ_ERR_NULL;
    if (misaligned(codes) || misaligned(sf) || misaligned(wq_packed) || misaligned(s_packed)) return NQ_ERR_ALIGN;
    const size_t cb = packed_bytes(kFp4, K, N), sb = scale_bytes(K, N, kFp4);
    const void* outs[2] = {wq_packed, s_packed};
    const size_t out_n[2] = {cb, sb};
    for (int i = 0; i < 2; ++i)
        if (overlap(outs[i], out_n[i], codes, cb) || overlap(outs[i], out_n[i], sf, sb)) return NQ_ERR_ALIAS;
    if (overlap(wq_packed, cb, s_packed, sb)) return NQ_ERR_ALIAS;
    DevState* d = nullptr;
    st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    const long long lanes = (long long)(N / kTileRows) * (K / kGroup) * 32;
    pack_fp4_codes_kernel<<<grid_for(lanes, 256), 256, 0, as_stream(stream)>>>(codes, K, N,
                                                                               static_cast<uint8_t*>(wq_packed));
    if (cudaGetLastError() != cudaSuccess) return NQ_ERR_CUDA;
    pack_fp4_scales_kernel<<<grid_for(lanes * 2, 256), 256, 0, as_stream(stream)>>>(sf, K, N,
                                                                                    static_cast<uint8_t*>(s_packed));
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

nq_status dequant_fp4(const void* wq, const void* sq, float gs, float* w, int K, int N, void* stream) {
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    if (K == 0 || N == 0) return NQ_OK;
    if (!wq || !sq || !w) return NQ_ERR_NULL;
    if (misaligned(wq) || misaligned(sq) || misaligned(w)) return NQ_ERR_ALIGN;
    if (overlap(w, (size_t)N * K * 4, wq, packed_bytes(kFp4, K, N)) ||
        overlap(w, (size_t)N * K * 4, sq, scale_bytes(K, N, kFp4)))
        return NQ_ERR_ALIAS;
    DevState* d = nullptr;
    st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    const long long lanes = (long long)(N / kTileRows) * (K / kGroup) * 32;
    dequant_fp4_kernel<<<grid_for(lanes, 256), 256, 0, as_stream(stream)>>>(
        static_cast<const uint8_t*>(wq), static_cast<const uint8_t*>(sq), gs, K, N, w);
    return cudaGetLastError() == cudaSuccess ? NQ_OK : NQ_ERR_CUDA;
}

}  // namespace

namespace nq {
unsigned long long wait_limit_ns() {
    std::lock_guard<std::mutex> lk(g_mu);
    read_env_locked();
    return g_wait_ns;
}

int check_projection_args(int bits, bool swiglu, const void* X, const void* W0, const void* S0, const void* W1,
                          const void* S1, const void* Y, int T, int K, int N) {
    return projection_args(bits, swiglu, X, W0, S0, W1, S1, Y, T, K, N);
}

int check_grouped_args(int bits, const void* X, const nq_group* groups, int count, int T, int K) {
    return grouped_args(bits, X, groups, count, T, K);
}

int reserve_projection_workspace(int bits, bool swiglu, int T, int K, int N) {
    return reserve_projection(bits, swiglu, T, K, N);
}

int reserve_grouped_workspace(int bits, const nq_group* groups, int count, int T, int K) {
    return reserve_grouped(bits, groups, count, T, K);
}

unsigned long long workspace_epoch() { return g_ws_epoch.load(); }
}  // namespace nq

// ---------------------------------------------------------------- C ABI

extern "C" {

const char* nq_status_string(nq_status s) {
    switch (s) {
        case NQ_OK: return "NQ_OK";
        case NQ_ERR_NULL: return "NQ_ERR_NULL: a required pointer is NULL";
        case NQ_ERR_SHAPE: return "NQ_ERR_SHAPE: need K % 64 == 0, N % 16 == 0, 0 <= T <= 64";
        case NQ_ERR_ALIGN: return "NQ_ERR_ALIGN: pointers must be 16-byte aligned";
        case NQ_ERR_ALIAS: return "NQ_ERR_ALIAS: an output overlaps an input";
        case NQ_ERR_CUDA: return "NQ_ERR_CUDA: a CUDA call or launch failed";
        case NQ_ERR_DEVICE: return "NQ_ERR_DEVICE: current device is not sm_103 (GB300)";
        case NQ_ERR_TIMEOUT: return "NQ_ERR_TIMEOUT: a bounded device-side wait ran out";
        case NQ_ERR_SCRATCH: return "NQ_ERR_SCRATCH: problem exceeds the fixed scratch of nq_gemm_q4_noalloc";
        default: return "NQ_ERR_UNKNOWN";
    }
}

int nq_version(void) { return (2 << 16) | 0; }

size_t nq_packed_bytes_q4(int K, int N) { return check_shape(K, N) == NQ_OK ? packed_bytes(4, K, N) : 0; }
size_t nq_packed_bytes_q5(int K, int N) { return check_shape(K, N) == NQ_OK ? packed_bytes(5, K, N) : 0; }

size_t nq_scale_bytes(int K, int N) { return check_shape(K, N) == NQ_OK ? scale_bytes(K, N) : 0; }
size_t nq_packed_bytes_fp4(int K, int N) { return check_shape(K, N) == NQ_OK ? packed_bytes(kFp4, K, N) : 0; }
size_t nq_scale_bytes_fp4(int K, int N) { return check_shape(K, N) == NQ_OK ? scale_bytes(K, N, kFp4) : 0; }

nq_status nq_pack_fp4(const uint32_t* codes_canon, const uint8_t* sf_canon, int K, int N, void* wq_packed,
                      void* s_packed, void* stream) {
    return pack_fp4(codes_canon, sf_canon, K, N, wq_packed, s_packed, stream);
}

nq_status nq_gemm_fp4(const void* X, const void* Wq, const void* S, float global_scale, void* Y, int T, int K, int N,
                      void* stream) {
    return project(kFp4, false, X, Wq, S, nullptr, nullptr, Y, T, K, N, stream, global_scale);
}

nq_status nq_dequant_fp4_debug(const void* Wq, const void* S, float global_scale, float* W, int K, int N,
                               void* stream) {
    return dequant_fp4(Wq, S, global_scale, W, K, N, stream);
}

nq_status nq_pack_q4(const uint32_t* wq_canon, const uint16_t* s_canon, int K, int N, void* wq_packed,
                     void* s_packed, void* stream) {
    return pack(4, wq_canon, nullptr, s_canon, K, N, wq_packed, s_packed, stream);
}

nq_status nq_pack_q5(const uint32_t* wn_canon, const uint32_t* wh_canon, const uint16_t* s_canon, int K, int N,
                     void* wq_packed, void* s_packed, void* stream) {
    return pack(5, wn_canon, wh_canon, s_canon, K, N, wq_packed, s_packed, stream);
}

nq_status nq_gemm_q4(const void* X, const void* Wq, const void* S, void* Y, int T, int K, int N, void* stream) {
    return project(4, false, X, Wq, S, nullptr, nullptr, Y, T, K, N, stream);
}

nq_status nq_gemm_q5(const void* X, const void* Wq, const void* S, void* Y, int T, int K, int N, void* stream) {
    return project(5, false, X, Wq, S, nullptr, nullptr, Y, T, K, N, stream);
}

nq_status nq_gemm_q4_grouped(const void* X, const nq_group* groups, int count, int T, int K, void* stream) {
    return project_grouped(4, X, groups, count, T, K, stream);
}

nq_status nq_gemm_q5_grouped(const void* X, const nq_group* groups, int count, int T, int K, void* stream) {
    return project_grouped(5, X, groups, count, T, K, stream);
}

nq_status nq_swiglu_q4(const void* X, const void* Wg, const void* Sg, const void* Wu, const void* Su, void* H, int T,
                       int K, int N, void* stream) {
    return project(4, true, X, Wg, Sg, Wu, Su, H, T, K, N, stream);
}

nq_status nq_swiglu_q5(const void* X, const void* Wg, const void* Sg, const void* Wu, const void* Su, void* H, int T,
                       int K, int N, void* stream) {
    return project(5, true, X, Wg, Sg, Wu, Su, H, T, K, N, stream);
}

nq_status nq_swiglu_fp4(const void* X, const void* Wg, const void* Sg, float gate_scale, const void* Wu,
                        const void* Su, float up_scale, void* H, int T, int K, int N, void* stream) {
    return project(kFp4, true, X, Wg, Sg, Wu, Su, H, T, K, N, stream, gate_scale, up_scale);
}

nq_status nq_dequant_q4_debug(const void* Wq, const void* S, float* W, int K, int N, void* stream) {
    return dequant(4, true, Wq, S, W, K, N, stream);
}

nq_status nq_dequant_q5_debug(const void* Wq, const void* S, float* W, int K, int N, void* stream) {
    return dequant(5, true, Wq, S, W, K, N, stream);
}

nq_status nq_dequant_q4_debug_bf16(const void* Wq, const void* S, float* W, int K, int N, void* stream) {
    return dequant(4, false, Wq, S, W, K, N, stream);
}

nq_status nq_dequant_q5_debug_bf16(const void* Wq, const void* S, float* W, int K, int N, void* stream) {
    return dequant(5, false, Wq, S, W, K, N, stream);
}

long long nq_wait_limit(long long ns) {
    std::lock_guard<std::mutex> lk(g_mu);
    read_env_locked();
    const long long prev = (long long)g_wait_ns;
    if (ns > 0) g_wait_ns = (unsigned long long)ns;
    return prev;
}

nq_status nq_reserve(int T_max, int K_max, int N_max) {
    if (T_max < 1 || T_max > kMaxT) return NQ_ERR_SHAPE;
    nq_status st = check_shape(K_max, N_max);
    if (st != NQ_OK) return st;
    DevState* d = nullptr;
    st = current_device(&d, nullptr);
    if (st != NQ_OK) return st;
    if (T_max > kSliceT) {
        // The tensor-core kernel's partials and tickets, for every shape up to the bound: a
        // plan has at most max(SMs, row blocks) blocks of kTcRows x TP partial floats and one
        // ticket per row block (reserved whether or not tensor-core batches are on now).
        const long long rb = ((N_max > 0 ? N_max : 16) + kTcRows - 1) / kTcRows;
        const long long blocks = rb > d->sms ? rb : d->sms;
        st = ensure_tc_workspace(*d, rb, blocks * kTcRows * tc_tpad(T_max));
        if (st != NQ_OK) return st;
        st = ensure_tc_gate(*d, (long long)T_max * (N_max > 0 ? N_max : 16));  // SwiGLU gate outputs
        if (st != NQ_OK) return st;
        T_max = kSliceT;  // the 8-token kernel's plans: slices of at most kSliceT tokens
    }
    long long slots = 0, tickets = 0;
    // The largest plan over T <= T_max and both modes bounds every smaller call; slab-cluster
    // plans (at most SMs / S clusters) are counted as well.
    for (int T = 1; T <= T_max; ++T)
        for (int mode = 0; mode < 2; ++mode) {
            const int K = K_max > 0 ? K_max : 64, N = N_max > 0 ? N_max : 16;
            Plan p;
            make_plan(4, mode, T, K, N, d->sms, p);
            if (p.slots > slots) slots = p.slots;
            if (p.RP > tickets) tickets = p.RP;
            Plan pc, qc;
            if (p.S >= 2 && p.S <= kMaxCluster && make_cluster_plans(4, mode, T, K, N, d->sms / p.S, pc, qc) &&
                qc.slots > slots)
                slots = qc.slots;
        }
    return ensure_workspace(*d, slots, tickets);
}

nq_status nq_device_error(void) {
    DevState* d = nullptr;
    int dev = 0;
    nq_status st = current_device(&d, &dev);
    if (st != NQ_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return NQ_ERR_CUDA;
    // The fixed scratch of nq_gemm_q4_noalloc has its own error word.
    const nq_status st_static = noalloc_take_error(dev);
    if (st_static == NQ_ERR_CUDA) return st_static;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!d->ws) return st_static;
    int err = 0;
    if (cudaMemcpy(&err, d->ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NQ_ERR_CUDA;
    if (err == 0) return st_static;
    if (cudaMemset(d->ws, 0, ws_partials_off(d->tickets_cap)) != cudaSuccess ||
        (d->tc_ws && cudaMemset(d->tc_ws, 0, (size_t)d->tc_tickets * 4) != cudaSuccess) ||
        cudaDeviceSynchronize() != cudaSuccess)
        return NQ_ERR_CUDA;
    return NQ_ERR_TIMEOUT;
}

void nq_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (int i = 0; i < kMaxDevices; ++i) {
        if (!g_dev[i].ws && !g_dev[i].tc_ws && !g_dev[i].tc_gate) continue;
        cudaSetDevice(i);
        cudaDeviceSynchronize();
        cudaFree(g_dev[i].ws);
        g_dev[i].ws = nullptr;
        g_dev[i].slots_cap = g_dev[i].tickets_cap = 0;
        cudaFree(g_dev[i].tc_ws);
        g_dev[i].tc_ws = nullptr;
        g_dev[i].tc_tickets = g_dev[i].tc_floats = 0;
        cudaFree(g_dev[i].tc_gate);
        g_dev[i].tc_gate = nullptr;
        g_dev[i].tc_gate_floats = 0;
        ++g_ws_epoch;
    }
    cudaSetDevice(cur);
}

nq_status nq_plan_info(int bits, int mode, int T, int K, int N, int num_sms, int64_t out[8]) {
    if (!out) return NQ_ERR_NULL;
    if ((bits != 4 && bits != 5) || (mode != 0 && mode != 1)) return NQ_ERR_SHAPE;
    if (T < 1 || T > 8 || K < kGroup || N < kTileRows || num_sms < 1) return NQ_ERR_SHAPE;
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    Plan p;
    if (!make_plan(bits, mode, T, K, N, num_sms, p)) return NQ_ERR_SHAPE;
    out[0] = p.P;
    out[1] = p.U;
    out[2] = p.S;
    out[3] = p.GS;
    out[4] = p.RP;
    out[5] = p.slots;
    out[6] = p.stages;
    out[7] = p.CG;
    return NQ_OK;
}

int64_t nq_plan_segments(int bits, int mode, int T, int K, int N, int num_sms, int cta, int64_t* seg,
                         int64_t cap) {
    int64_t info[8];
    nq_status st = nq_plan_info(bits, mode, T, K, N, num_sms, info);
    if (st != NQ_OK) return st;
    Plan p;
    make_plan(bits, mode, T, K, N, num_sms, p);
    if (cta < 0 || cta >= p.P) return NQ_ERR_SHAPE;
    if (cap > 0 && !seg) return NQ_ERR_NULL;
    // Same walk as the kernels: the block's segments in processing order.
    int64_t n = 0;
    const long long u0 = cta_begin(p, cta), u1 = cta_begin(p, cta + 1);
    const SegOrder order = seg_order(p, u0, u1);
    Segment nat;
    for (int si = 0; si < order.count; ++si) {
        const Segment sg = seg_pick(p, order, si, nat, u1);
        if (n < cap) {
            seg[4 * n + 0] = sg.s;
            seg[4 * n + 1] = sg.rp;
            seg[4 * n + 2] = sg.ga;
            seg[4 * n + 3] = sg.gb;
        }
        ++n;
    }
    return n;
}

int nq_tensor_core_batches(int enable) {
    DevState* d = nullptr;
    current_device(&d, nullptr);  // reads the environment once, like every call
    std::lock_guard<std::mutex> lk(g_mu);
    const int prev = g_tc ? 1 : 0;
    if (enable == 0 || enable == 1) g_tc = enable == 1;
    return prev;
}

nq_status nq_plan_tc_info(int bits, int T, int K, int N, int num_sms, int64_t out[8]) {
    if (!out) return NQ_ERR_NULL;
    if ((bits != 4 && bits != 5 && bits != kFp4) || T <= kSliceT || T > kTcMaxT || num_sms < 1 || K < kGroup ||
        N < kTileRows)
        return NQ_ERR_SHAPE;
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    TcPlan p;
    if (!make_tc_plan(bits, T, K, N, num_sms, p)) return NQ_ERR_SHAPE;
    out[0] = p.P;
    out[1] = p.RB;
    out[2] = p.KS;
    out[3] = p.TP;
    out[4] = p.stages;
    out[5] = p.smem_bytes;
    out[6] = p.G;
    out[7] = tc_stage_groups(p.TP);
    return NQ_OK;
}

nq_status nq_route_info(int bits, int mode, int T, int K, int N, int num_sms, int64_t out[8]) {
    if (!out) return NQ_ERR_NULL;
    if ((bits != 4 && bits != 5 && bits != kFp4) || (mode != 0 && mode != 1)) return NQ_ERR_SHAPE;
    if (T < 1 || T > kMaxT || K < kGroup || N < kTileRows || num_sms < 1) return NQ_ERR_SHAPE;
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    bool tc = true, cluster = false;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        read_env_locked();
        tc = g_tc;
        cluster = g_cluster;
    }
    // the branch project() takes: the tensor-core kernel for 8 < T <= 64 ...
    if (tc && T > kSliceT && T <= kTcMaxT) {
        TcPlan p;
        if (make_tc_plan(bits, T, K, N, num_sms, p)) {
            out[0] = 1;
            out[1] = mode == 1 ? 2 : 1;
            out[2] = 1;
            out[3] = 3;
            out[4] = p.P;
            out[5] = p.KS;
            out[6] = p.stages;
            out[7] = p.TP;
            return NQ_OK;
        }
    }
    // ... else one launch of the 8-token kernel per slice of up to 8 tokens (the first slice's
    // plan), slab clusters when switched on and K needs 2..4 bf16 slabs (assuming every
    // cluster the SMs hold is resident)
    const int full = T < kSliceT ? T : kSliceT;
    Plan p;
    if (!make_plan(bits, mode, full, K, N, num_sms, p)) return NQ_ERR_SHAPE;
    int split = p.S == 1 && p.U % p.P == 0 && (p.U / p.P) % p.G == 0 ? 1 : 0;
    if (cluster && p.S >= 2 && p.S <= kMaxCluster && !p.f16) {
        Plan pc, qc;
        if (make_cluster_plans(bits, mode, full, K, N, num_sms / p.S, pc, qc)) {
            p = pc;
            split = 2;
        }
    }
    out[0] = 0;
    out[1] = (T + kSliceT - 1) / kSliceT;
    out[2] = p.f16 ? 0 : 1;
    out[3] = split;
    out[4] = p.P;
    out[5] = p.S;
    out[6] = p.stages;
    out[7] = p.TP;
    return NQ_OK;
}

int nq_slab_clusters(int enable) {
    DevState* d = nullptr;
    current_device(&d, nullptr);  // reads the environment once, like every call
    std::lock_guard<std::mutex> lk(g_mu);
    const int prev = g_cluster ? 1 : 0;
    if (enable == 0 || enable == 1) g_cluster = enable == 1;
    return prev;
}

nq_status nq_plan_cluster_info(int bits, int mode, int T, int K, int N, int clusters, int64_t out[8]) {
    if (!out) return NQ_ERR_NULL;
    if ((bits != 4 && bits != 5) || (mode != 0 && mode != 1)) return NQ_ERR_SHAPE;
    if (T < 1 || T > 8 || K < kGroup || N < kTileRows || clusters < 1) return NQ_ERR_SHAPE;
    nq_status st = check_shape(K, N);
    if (st != NQ_OK) return st;
    Plan p, q;
    if (!make_cluster_plans(bits, mode, T, K, N, clusters, p, q)) return NQ_ERR_SHAPE;
    out[0] = p.P;
    out[1] = p.cl;
    out[2] = p.GS;
    out[3] = p.RP;
    out[4] = q.slots;
    out[5] = p.stages;
    out[6] = q.U;
    out[7] = q.P;
    return NQ_OK;
}

int64_t nq_plan_cluster_segments(int bits, int mode, int T, int K, int N, int clusters, int cta, int64_t* seg,
                                 int64_t cap) {
    int64_t info[8];
    nq_status st = nq_plan_cluster_info(bits, mode, T, K, N, clusters, info);
    if (st != NQ_OK) return st;
    Plan p, q;
    make_cluster_plans(bits, mode, T, K, N, clusters, p, q);
    if (cta < 0 || cta >= p.P) return NQ_ERR_SHAPE;
    if (cap > 0 && !seg) return NQ_ERR_NULL;
    // Same walk as the kernels: the cluster's segments in processing order, mapped to the
    // block's rank (its slab).
    const int c = cta / p.cl, r = cta % p.cl;
    int64_t n = 0;
    const long long u0 = cta_begin(q, c), u1 = cta_begin(q, c + 1);
    const SegOrder order = seg_order(q, u0, u1);
    Segment nat;
    for (int si = 0; si < order.count; ++si) {
        const Segment sg = rank_segment(p, seg_pick(q, order, si, nat, u1), r);
        if (n < cap) {
            seg[4 * n + 0] = sg.s;
            seg[4 * n + 1] = sg.rp;
            seg[4 * n + 2] = sg.ga;
            seg[4 * n + 3] = sg.gb;
        }
        ++n;
    }
    return n;
}

}  // extern "C"
