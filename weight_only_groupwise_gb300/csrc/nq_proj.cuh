// nq_proj.cuh -- the projection kernel: Y[T,N] = X[T,K] * dequant(W) for T <= 8, 4- or 5-bit
// codes with one fp16 scale per 64-wide K group, optionally fused into the SwiGLU gate/up
// pair ("NInfer-4090" release post, section "V3 做了什么": small-batch Q4/Q5 projections
// tuned at T=8 for GDN, attention and SwiGLU; "ninfer-ext" README, section
// "与原版 NInfer 的对比": the Q5 K-split MMA path for verify rounds).
//
// Structure (one persistent block per SM, 8 consumer warps + 1 producer warp):
//   * The producer's elected lane streams the block's contiguous range of packed tiles with
//     1-D TMA bulk copies into a ring of shared-memory stages (mbarrier full/empty pairs,
//     L2 evict-first: every weight byte is read exactly once). It also bulk-copies the
//     activations of the current K slab (T rows, padded) into shared memory.
//   * Consumer warps split each stage's K groups. Per group and 16-row tile a lane decodes
//     its 16 code bytes into bf16 A fragments holding 128 + q (exact), loads the B fragment
//     of X with ldmatrix, and runs four m16n8k16 MMAs whose accumulator starts at
//     -(128 + z) * sum(x) of the group -- so the group partial is exactly sum((q - z) * x) up
//     to fp32 rounding -- then applies the fp16 scale with one FMA into the fp32 accumulator.
//   * At the end of each (slab, row pair) run the warps reduce through shared memory in a
//     fixed order. A run owned entirely by one block writes Y directly. Otherwise the block
//     stores an fp32 partial in the workspace and takes a ticket; the block that takes the
//     last ticket sums all partials of the pair in a fixed order (deterministic split-K,
//     no spinning on other blocks) and writes Y.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "nq_common.cuh"

namespace nq {

struct ProjArgs {
    const uint16_t* X;   // bf16 [T][K]
    const uint8_t* W0;   // packed codes of M tile 0's matrix
    const uint8_t* S0;   // packed scales of M tile 0's matrix
    const uint8_t* W1;   // M tile 1 (gemm: same matrix, next row tile; swiglu: up matrix)
    const uint8_t* S1;
    uint16_t* Y;         // bf16 [T][N]
    float* partials;     // workspace: slots x kPartialFloats
    int* tickets;        // workspace: one per row pair, zero between calls
    int* dev_err;        // workspace: device error word
    Plan p;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Shared-memory row pitch of one activation row of a slab: 16 bytes of padding make the 8
// token rows of an ldmatrix phase fall on distinct bank groups.
__host__ __device__ __forceinline__ int x_pitch(int gs) { return gs * 128 + 16; }

// One 16-row x 64-K tile: decode, 4 MMAs, scale. xb = B fragments of the 4 K steps,
// (c0, c1) = (128 + z) * sum(x) of this group for the lane's two token columns.
// (128 + q) - (128 + z) on bf16x2 pairs: exact, the result q - z is a small integer.
template <int BITS>
__device__ __forceinline__ void to_signed(uint32_t a[4]) {
    const __nv_bfloat162 off = __floats2bfloat162_rn(BITS == 4 ? 136.0f : 144.0f, BITS == 4 ? 136.0f : 144.0f);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&a[m]);
        v = __hsub2(v, off);
        a[m] = *reinterpret_cast<uint32_t*>(&v);
    }
}

// One K step: decode word J of the lane into the A fragment, then MMA.
template <int BITS, bool FOLD, int J>
__device__ __forceinline__ void step_mma(float d[4], uint32_t w, uint32_t hb, uint32_t b0, uint32_t b1) {
    uint32_t af[4];
    if constexpr (BITS == 4) decode_q4(w, af); else decode_q5<J>(w, hb, af);
    if constexpr (!FOLD) to_signed<BITS>(af);
    mma_bf16_16816(d, af, b0, b1);
}

// FOLD: A holds 128 + q and the accumulator starts at -(c0, c1) = -(128 + z) * sum(x);
// otherwise A holds the exact q - z and the accumulator starts at zero.
template <int BITS, bool FOLD>
__device__ __forceinline__ void tile_mma(const uint8_t* tile, const uint8_t* sc, int lane,
                                         const uint32_t xb[8], float c0, float c1, float acc[4]) {
    const uint4 w = *reinterpret_cast<const uint4*>(tile + lane * 16);
    uint32_t hb = 0;
    if constexpr (BITS == 5) hb = *reinterpret_cast<const uint32_t*>(tile + 512 + lane * 4);
    const uint32_t sw = *reinterpret_cast<const uint32_t*>(sc + (lane >> 2) * 4);
    float d[4] = {-c0, -c1, -c0, -c1};
    step_mma<BITS, FOLD, 0>(d, w.x, hb, xb[0], xb[1]);
    step_mma<BITS, FOLD, 1>(d, w.y, hb, xb[2], xb[3]);
    step_mma<BITS, FOLD, 2>(d, w.z, hb, xb[4], xb[5]);
    step_mma<BITS, FOLD, 3>(d, w.w, hb, xb[6], xb[7]);
    __half2 sh;
    *reinterpret_cast<uint32_t*>(&sh) = sw;
    const float2 s = __half22float2(sh);
    acc[0] = fmaf(s.x, d[0], acc[0]);
    acc[1] = fmaf(s.x, d[1], acc[1]);
    acc[2] = fmaf(s.y, d[2], acc[2]);
    acc[3] = fmaf(s.y, d[3], acc[3]);
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

template <int BITS, bool SWIGLU, bool FOLD>
__global__ void __launch_bounds__(kThreads, 1) proj_kernel(const __grid_constant__ ProjArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const Plan& p = a.p;
    constexpr int TB = BITS == 4 ? kQ4TileBytes : kQ5TileBytes;
    constexpr float kOffset = BITS == 4 ? 136.0f : 144.0f;  // 128 + z
    constexpr int kConsumers = kConsumerWarps * 32;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;

    uint8_t* stage_mem = smem;
    uint8_t* xs = smem + p.stages * p.stage_bytes;
    float* corr = reinterpret_cast<float*>(xs + p.x_bytes);
    float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(corr) + p.corr_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + p.red_bytes);
    // bars: full[kMaxStages], empty[kMaxStages]; then x_full, x_empty; then flags
    volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages + 2);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
    const uint32_t x_full = smem_u32(bars + 2 * kMaxStages), x_empty = x_full + 8;
    // zero row for ldmatrix lanes of absent tokens: the 16 bytes after the last X row
    const int pitch = x_pitch(p.GS);
    uint8_t* zero_row = xs + p.T * pitch;

    if (tid == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kConsumerWarps);
        }
        mbar_init(x_full, 1);
        mbar_init(x_empty, kConsumerWarps);
        flags[0] = 0;  // abort
        flags[1] = 0;  // last-arriver broadcast
        *reinterpret_cast<uint4*>(zero_row) = make_uint4(0, 0, 0, 0);
        mbar_fence_init();
    }
    __syncthreads();
    // Programmatic dependent launch: nothing below touches global memory that the
    // preceding kernel in the stream may still write before this point.
    grid_dependency_wait();
    // Let the next kernel in the stream be scheduled as SMs free up; it waits in turn.
    grid_launch_dependents();

    const long long u0 = cta_begin(p, cta), u1 = cta_begin(p, cta + 1);

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int it = 0, nx = 0, cur_slab = -1;
            bool ok = true;
            for (long long u = u0; u < u1 && ok;) {
                const Segment sg = segment_at(p, u, u1);
                if (sg.s != cur_slab) {
                    if (!mbar_wait(x_empty, (nx & 1) ^ 1, flags, a.dev_err)) { ok = false; break; }
                    const int gs = slab_groups(p, sg.s);
                    const uint32_t row_bytes = gs * 128;
                    mbar_arrive_expect_tx(x_full, row_bytes * p.T);
                    for (int t = 0; t < p.T; ++t)
                        bulk_g2s_keep(smem_u32(xs + t * pitch),
                                      a.X + (size_t)t * p.K + (size_t)sg.s * p.GS * kGroup, row_bytes,
                                      x_full);
                    ++nx;
                    cur_slab = sg.s;
                }
                const int rt0 = SWIGLU ? sg.rp : 2 * sg.rp;
                const int rt1 = SWIGLU ? sg.rp : 2 * sg.rp + 1;
                const bool has1 = SWIGLU || rt1 < p.RT;
                for (int ga = sg.ga; ga < sg.gb; ga += p.CG, ++it) {
                    const int n = min(p.CG, sg.gb - ga);
                    const int st = it % p.stages;
                    if (!mbar_wait(empty0 + 8 * st, ((it / p.stages) & 1) ^ 1, flags, a.dev_err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sb = stage_mem + st * p.stage_bytes;
                    const uint32_t cb = n * TB, sbytes = n * kScaleTileBytes;
                    const uint32_t fb = full0 + 8 * st;
                    mbar_arrive_expect_tx(fb, (has1 ? 2u : 1u) * (cb + sbytes));
                    bulk_g2s(smem_u32(sb), a.W0 + ((size_t)rt0 * p.G + ga) * TB, cb, fb, pol);
                    bulk_g2s(smem_u32(sb + 2 * p.CG * TB),
                             a.S0 + ((size_t)rt0 * p.G + ga) * kScaleTileBytes, sbytes, fb, pol);
                    if (has1) {
                        bulk_g2s(smem_u32(sb + p.CG * TB), a.W1 + ((size_t)rt1 * p.G + ga) * TB, cb,
                                 fb, pol);
                        bulk_g2s(smem_u32(sb + 2 * p.CG * TB + p.CG * kScaleTileBytes),
                                 a.S1 + ((size_t)rt1 * p.G + ga) * kScaleTileBytes, sbytes, fb, pol);
                    }
                }
                u = sg.u_next;
            }
            if (!ok) {
                // Aborted: let copies already issued land before the block can exit.
                const int first = it > p.stages ? it - p.stages : 0;
                for (int j = first; j < it; ++j)
                    mbar_wait_drain(full0 + 8 * (j % p.stages), (j / p.stages) & 1, 100000000ull);
                if (nx > 0) mbar_wait_drain(x_full, (nx - 1) & 1, 100000000ull);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    float acc[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[m][j] = 0.f;

    // ldmatrix row addresses: lane l serves row (l & 7) of matrix (l >> 3); matrix mi covers
    // K step (mi >> 1) and its half (mi & 1). Absent tokens read the zero row.
    const int lt = lane & 7, mi = lane >> 3;
    const bool lt_valid = lt < p.T;
    const uint32_t ld_base = lt_valid ? smem_u32(xs + lt * pitch + ((mi >> 1) * 16 + (mi & 1) * 8) * 2)
                                      : smem_u32(zero_row);
    const uint32_t ld_group_step = lt_valid ? 128u : 0u;
    const uint32_t ld_half_step = lt_valid ? 64u : 0u;  // K steps 2,3 are 32 elements further
    const int c4 = lane & 3;

    int it = 0, nx = 0, cur_slab = -1;
    for (long long u = u0; u < u1;) {
        const Segment sg = segment_at(p, u, u1);
        if (sg.s != cur_slab) {
            if (cur_slab >= 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(x_empty);
            }
            mbar_wait(x_full, nx & 1, flags, a.dev_err);
            ++nx;
            cur_slab = sg.s;
            // corr[gl][t] = (128 + z) * sum of the group's 64 activations of token t
            const int gs = slab_groups(p, sg.s);
            for (int task = tid; task < gs * 8; task += kConsumers) {
                const int gl = task >> 3, t = task & 7;
                float sum = 0.f;
                if (FOLD && t < p.T && !flags[0]) {
                    const uint4* row = reinterpret_cast<const uint4*>(xs + t * pitch + gl * 128);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const uint4 q = row[v];
                        sum += __uint_as_float(q.x << 16) + __uint_as_float(q.x & 0xFFFF0000u);
                        sum += __uint_as_float(q.y << 16) + __uint_as_float(q.y & 0xFFFF0000u);
                        sum += __uint_as_float(q.z << 16) + __uint_as_float(q.z & 0xFFFF0000u);
                        sum += __uint_as_float(q.w << 16) + __uint_as_float(q.w & 0xFFFF0000u);
                    }
                }
                corr[task] = kOffset * sum;
            }
            named_bar_sync(1, kConsumers);
        }

        const int rt1 = SWIGLU ? sg.rp : 2 * sg.rp + 1;
        const bool has1 = SWIGLU || rt1 < p.RT;
        const int slab_g0 = sg.s * p.GS;
        for (int ga = sg.ga; ga < sg.gb; ga += p.CG, ++it) {
            const int n = min(p.CG, sg.gb - ga);
            const int st = it % p.stages;
            const bool ok = mbar_wait(full0 + 8 * st, (it / p.stages) & 1, flags, a.dev_err);
            if (ok) {
                const uint8_t* sb = stage_mem + st * p.stage_bytes;
                const uint8_t* sc0 = sb + 2 * p.CG * TB;
                for (int i = warp; i < n; i += kConsumerWarps) {
                    const int gl = ga + i - slab_g0;
                    uint32_t xb[8];
                    const uint32_t la = ld_base + gl * ld_group_step;
                    ldsm_x4(la, xb);
                    ldsm_x4(la + ld_half_step, xb + 4);
                    const float2 cr = *reinterpret_cast<const float2*>(corr + gl * 8 + 2 * c4);
                    tile_mma<BITS, FOLD>(sb + i * TB, sc0 + i * kScaleTileBytes, lane, xb, cr.x, cr.y, acc[0]);
                    if (has1)
                        tile_mma<BITS, FOLD>(sb + p.CG * TB + i * TB,
                                       sc0 + p.CG * kScaleTileBytes + i * kScaleTileBytes, lane, xb,
                                       cr.x, cr.y, acc[1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }

        // ------------------------------------------------------------ run epilogue
        {
            float4* r4 = reinterpret_cast<float4*>(red);
            r4[(warp * 2 + 0) * 32 + lane] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
            r4[(warp * 2 + 1) * 32 + lane] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[m][j] = 0.f;
            named_bar_sync(1, kConsumers);

            // thread -> (tile m, token, row); output index o = m*128 + tok*16 + row
            const int m = SWIGLU ? 0 : (tid >> 7);
            const int r = tid & 127;
            const int tok = r >> 4, row = r & 15;
            const int l = (row & 7) * 4 + (tok >> 1), j = (row >> 3) * 2 + (tok & 1);
            const bool active = SWIGLU ? tid < 128 : true;
            float v0 = 0.f, v1 = 0.f;
            if (active) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    v0 += red[((w * 2 + m) * 32 + l) * 4 + j];
                    if (SWIGLU) v1 += red[((w * 2 + 1) * 32 + l) * 4 + j];
                }
            }
            const int rt = SWIGLU ? sg.rp : 2 * sg.rp + m;
            const bool out_ok = active && tok < p.T && rt < p.RT;
            const size_t yi = (size_t)tok * p.N + (size_t)rt * kTileRows + row;
            const int fan_in = contributions(p, sg.rp);
            if (fan_in == 1) {
                if (out_ok && !flags[0])
                    a.Y[yi] = SWIGLU ? bf16_bits_rn(silu_mul(v0, v1)) : bf16_bits_rn(v0);
            } else {
                float* ws = a.partials + slot_of(p, sg.s, sg.rp, cta) * kPartialFloats;
                if (active) {
                    ws[tid] = v0;
                    if (SWIGLU) ws[128 + tid] = v1;
                }
                __threadfence();
                named_bar_sync(1, kConsumers);
                if (tid == 0) {
                    int last = 0;
                    if (!flags[0]) last = atomicAdd(a.tickets + sg.rp, 1) == fan_in - 1;
                    flags[1] = last;
                }
                named_bar_sync(1, kConsumers);
                if (flags[1]) {
                    __threadfence();
                    float s0 = 0.f, s1 = 0.f;
                    for (int s = 0; s < p.S; ++s) {
                        const int gs = slab_groups(p, s);
                        const long long r0 = slab_base(p, s) + (long long)sg.rp * gs;
                        const int c_end = cta_of(p, r0 + gs - 1);
                        for (int c = cta_of(p, r0); c <= c_end; ++c) {
                            const float* src = a.partials + slot_of(p, s, sg.rp, c) * kPartialFloats;
                            if (active) {
                                s0 += __ldcg(src + tid);
                                if (SWIGLU) s1 += __ldcg(src + 128 + tid);
                            }
                        }
                    }
                    if (out_ok) a.Y[yi] = SWIGLU ? bf16_bits_rn(silu_mul(s0, s1)) : bf16_bits_rn(s0);
                    if (tid == 0) a.tickets[sg.rp] = 0;
                }
            }
            named_bar_sync(1, kConsumers);
        }
        u = sg.u_next;
    }

    if (flags[0] && tid == 0) {
        // Aborted: wait (bounded) for any stage copies still in flight before exiting.
        const int first = it > p.stages ? it - p.stages : 0;
        for (int j = first; j < it; ++j)
            mbar_wait_drain(full0 + 8 * (j % p.stages), (j / p.stages) & 1, 100000000ull);
    }
}

}  // namespace nq
