// nq_proj.cuh -- the projection kernel: Y[T,N] = X[T,K] * dequant(W) for T <= 8, 4- or 5-bit
// codes with one fp16 scale per 64-wide K group, optionally fused into the SwiGLU gate/up
// pair ("NInfer-4090" release post, section "V3 做了什么": small-batch Q4/Q5 projections
// tuned at T=8 for GDN, attention and SwiGLU; "ninfer-ext" README, section
// "与原版 NInfer 的对比": the Q5 K-split MMA path for verify rounds).
//
// Structure: one persistent block per SM with three roles.
//   * Producer warp: its elected lane streams the block's units with 1-D TMA bulk copies
//     into a ring of shared-memory stages (mbarrier full/empty pairs, L2 evict-first: every
//     weight byte is read exactly once). A stage holds one 16-group packed block (codes and
//     scales) of each of the two M tiles: one copy per tile, which keeps the copy engine at
//     full rate. It also bulk-copies the activations of the current K slab (T rows, padded).
//   * Consumer warps (kConsumerWarps): warp w takes K groups w and w + 8 of every stage, for
//     both 16-row tiles of the row pair. A lane decodes its 16 code bytes into bf16 A
//     fragments holding 128 + q (exact), loads the B fragment of X with ldmatrix and runs
//     four m16n8k16 MMAs from a zero accumulator: P = sum((128 + q) * x). The MMAs of the
//     warp's four tiles are issued K-step by K-step so the four accumulator chains overlap.
//     The same four MMAs on the constant code z give O = sum((128 + z) * x) once per group
//     and slab; P - O = sum((q - z) * x) up to fp32 rounding, and exactly 0 where every code
//     equals z (identical MMA inputs). The fp16 scale is applied with one FMA per group.
//   * Epilogue warp: at the end of each (slab, row pair) run the consumers drop their
//     accumulators into one of two shared buffers and carry on. The epilogue warp reduces
//     the warps' parts in a fixed order and writes Y directly when the run covers its whole
//     pair; otherwise it stores an fp32 partial in the workspace and takes a ticket; the
//     block that takes the last ticket sums all partials of the pair in a fixed order
//     (deterministic split-K, no spinning on other blocks) and writes Y. The block's
//     partial runs are processed first, so split-K settles early and the block ends on a
//     complete run.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "nq_common.cuh"

namespace nq {

struct ProjArgs {
    const uint16_t* X;   // bf16 [T][K]
    const uint8_t* W0;   // packed matrix of M tile 0 (codes and scales)
    const uint8_t* W1;   // M tile 1 (gemm: same matrix, next row tile; swiglu: up matrix)
    uint16_t* Y;         // bf16 [T][N]
    float* partials;     // workspace: slots x kPartialFloats
    int* tickets;        // workspace: one per row pair, zero between calls
    int* dev_err;        // workspace: device error word
    Plan p;
};

// Named barriers: 1 = consumers only; 2,3 = run buffer b full (consumers arrive, epilogue
// syncs); 4,5 = run buffer b free (epilogue arrives, consumers sync).
constexpr int kBarConsumers = 1, kBarRedFull = 2, kBarRedFree = 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kHandoffThreads = kConsumerThreads + 32;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Shared-memory row pitch of one activation row of a slab: 16 bytes of padding make the 8
// token rows of an ldmatrix phase fall on distinct bank groups.
__host__ __device__ __forceinline__ int x_pitch(int gs) { return gs * 128 + 16; }

template <int J>
__device__ __forceinline__ uint32_t word_of(const uint4& w) {
    return J == 0 ? w.x : (J == 1 ? w.y : (J == 2 ? w.z : w.w));
}

// A fragment of K step J: 128 + q as bf16 pairs.
template <int BITS, int J>
__device__ __forceinline__ void decode_step(const uint4& w, uint32_t hb, uint32_t a[4], uint32_t magic) {
    if constexpr (BITS == 4) decode_q4(word_of<J>(w), a, magic);
    else decode_q5<J>(word_of<J>(w), hb, a, magic);
}

// Which group (0/1: B fragments xb[h], O o[h]) and which M tile (acc[m]) tile t of a pass
// uses. GROUPS groups x TILES M tiles, tile t = m * GROUPS + h.
template <int GROUPS>
__device__ __forceinline__ constexpr int group_of(int t) { return t % GROUPS; }
template <int GROUPS>
__device__ __forceinline__ constexpr int mtile_of(int t) { return t / GROUPS; }

// GROUPS x TILES tiles in one pass, K-step-major so their accumulator chains overlap. Each
// tile's chain is "zero, then K steps 0..3", exactly as for O. code[t] / scale[t]: this
// lane's code bytes / scale pair of tile t.
template <int BITS, int GROUPS, int TILES>
__device__ __forceinline__ void tiles_mma(const uint8_t* const (&code)[GROUPS * TILES],
                                          const uint8_t* const (&scale)[GROUPS * TILES],
                                          const uint32_t (&xb)[2][8], const float2 (&o)[2], uint32_t magic,
                                          float (&acc)[2][4]) {
    constexpr int NT = GROUPS * TILES;
    uint4 w[NT];
    uint32_t hb[NT], sw[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        w[t] = *reinterpret_cast<const uint4*>(code[t]);
        // high-bit word of the lane: after the tile's 512 nibble bytes, 4 bytes per lane
        hb[t] = BITS == 5 ? *reinterpret_cast<const uint32_t*>(code[t] + 512 - (threadIdx.x & 31) * 12) : 0u;
        sw[t] = *reinterpret_cast<const uint32_t*>(scale[t]);
    }
    float d[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) d[t][0] = d[t][1] = d[t][2] = d[t][3] = 0.f;
    uint32_t a[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) decode_step<BITS, 0>(w[t], hb[t], a[t], magic);
#pragma unroll
    for (int t = 0; t < NT; ++t) mma_bf16_16816(d[t], a[t], xb[group_of<GROUPS>(t)][0], xb[group_of<GROUPS>(t)][1]);
#pragma unroll
    for (int t = 0; t < NT; ++t) decode_step<BITS, 1>(w[t], hb[t], a[t], magic);
#pragma unroll
    for (int t = 0; t < NT; ++t) mma_bf16_16816(d[t], a[t], xb[group_of<GROUPS>(t)][2], xb[group_of<GROUPS>(t)][3]);
#pragma unroll
    for (int t = 0; t < NT; ++t) decode_step<BITS, 2>(w[t], hb[t], a[t], magic);
#pragma unroll
    for (int t = 0; t < NT; ++t) mma_bf16_16816(d[t], a[t], xb[group_of<GROUPS>(t)][4], xb[group_of<GROUPS>(t)][5]);
#pragma unroll
    for (int t = 0; t < NT; ++t) decode_step<BITS, 3>(w[t], hb[t], a[t], magic);
#pragma unroll
    for (int t = 0; t < NT; ++t) mma_bf16_16816(d[t], a[t], xb[group_of<GROUPS>(t)][6], xb[group_of<GROUPS>(t)][7]);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        __half2 sh;
        *reinterpret_cast<uint32_t*>(&sh) = sw[t];
        const float2 s = __half22float2(sh);
        const int m = mtile_of<GROUPS>(t), h = group_of<GROUPS>(t);
        acc[m][0] = fmaf(s.x, d[t][0] - o[h].x, acc[m][0]);
        acc[m][1] = fmaf(s.x, d[t][1] - o[h].y, acc[m][1]);
        acc[m][2] = fmaf(s.y, d[t][2] - o[h].x, acc[m][2]);
        acc[m][3] = fmaf(s.y, d[t][3] - o[h].y, acc[m][3]);
    }
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Output element (tile m, token, row) of a run -> its place in the consumers' accumulator
// layout (m16n8 C fragment: lane l holds rows l/4 and l/4+8, tokens 2(l%4) and 2(l%4)+1).
__device__ __forceinline__ int red_index(int w, int m, int tok, int row) {
    const int l = (row & 7) * 4 + (tok >> 1), j = (row >> 3) * 2 + (tok & 1);
    return ((w * 2 + m) * 32 + l) * 4 + j;
}

template <int BITS, bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1) proj_kernel(const __grid_constant__ ProjArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int TB = BITS == 4 ? kQ4TileBytes : kQ5TileBytes;
    constexpr int TBS = TB + kScaleTileBytes;         // code + scale bytes per tile
    constexpr int BG = kBlockGroups;                  // groups per block = per stage
    constexpr int kTileArea = BG * TBS;               // one M tile's share of a stage
    constexpr int kStageBytes = 2 * kTileArea;
    constexpr int NW = kConsumerWarps;
    constexpr int kRedFloats = NW * 2 * 128;          // one run buffer
    static_assert(kGroupsPerWarp == 2, "two groups per warp per stage");
    // bf16 pair of the zero-point code in the 128 + q encoding: 136 (Q4) or 144 (Q5)
    constexpr uint32_t kZeroCode = BITS == 4 ? 0x43084308u : 0x43104310u;

    // plan fields used in loops, in registers
    const Plan& p = a.p;
    const int T = p.T, G = p.G, RT = p.RT, GS = p.GS, nstages = p.stages;
    const long long row_tile_bytes = (long long)G * TBS;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;

    uint8_t* stage_mem = smem;
    uint8_t* xs = smem + nstages * kStageBytes;
    float* osum = reinterpret_cast<float*>(xs + p.x_bytes);  // O[gl][8]
    float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(osum) + p.corr_bytes);  // [2][kRedFloats]
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + p.red_bytes);
    // bars: full[kMaxStages], empty[kMaxStages]; then x_full, x_empty; then flags
    volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages + 2);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
    const uint32_t x_full = smem_u32(bars + 2 * kMaxStages), x_empty = x_full + 8;
    // zero row for ldmatrix lanes of absent tokens: the 16 bytes after the last X row
    const int pitch = x_pitch(GS);
    uint8_t* zero_row = xs + T * pitch;

    if (tid == 0) {
        for (int i = 0; i < nstages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kConsumerWarps);
        }
        mbar_init(x_full, 1);
        mbar_init(x_empty, kConsumerWarps);
        flags[0] = 0;  // abort
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
    const SegOrder order = seg_order(p, u0, u1);

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int it = 0, st = 0, nx = 0, cur_slab = -1;
            uint32_t phase = 0;
            bool ok = true;
            Segment nat;
            for (int si = 0; si < order.count && ok; ++si) {
                const Segment sg = seg_pick(p, order, si, nat, u1);
                if (sg.s != cur_slab) {
                    if (!mbar_wait(x_empty, (nx & 1) ^ 1, flags, a.dev_err)) { ok = false; break; }
                    const int gs = slab_groups(p, sg.s);
                    const uint32_t row_bytes = gs * 128;
                    mbar_arrive_expect_tx(x_full, row_bytes * T);
                    for (int t = 0; t < T; ++t)
                        bulk_g2s_keep(smem_u32(xs + t * pitch),
                                      a.X + (size_t)t * p.K + (size_t)sg.s * GS * kGroup, row_bytes, x_full);
                    ++nx;
                    cur_slab = sg.s;
                }
                const int rt0 = SWIGLU ? sg.rp : 2 * sg.rp;
                const int rt1 = SWIGLU ? sg.rp : 2 * sg.rp + 1;
                const bool has1 = SWIGLU || rt1 < RT;
                const uint8_t* w0 = a.W0 + rt0 * row_tile_bytes;
                const uint8_t* w1 = a.W1 + rt1 * row_tile_bytes;
                for (int b = sg.ga / BG; b * BG < sg.gb; ++b) {
                    const int i0 = max(sg.ga - b * BG, 0), i1 = min(sg.gb - b * BG, BG);
                    const int nb = block_groups(b, G);
                    const bool whole = i0 == 0 && i1 == BG;   // implies nb == BG
                    if (!mbar_wait(empty0 + 8 * st, phase ^ 1, flags, a.dev_err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sb = stage_mem + st * kStageBytes;
                    const uint32_t fb = full0 + 8 * st;
                    const uint32_t per_tile = (i1 - i0) * TBS;
                    mbar_arrive_expect_tx(fb, (has1 ? 2u : 1u) * per_tile);
                    const long long boff = (long long)b * BG * TBS;
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        if (m == 1 && !has1) break;
                        const uint8_t* blk = (m == 0 ? w0 : w1) + boff;
                        uint8_t* dst = sb + m * kTileArea;
                        if (whole) {
                            bulk_g2s(smem_u32(dst), blk, kTileArea, fb, pol);
                        } else {
                            bulk_g2s(smem_u32(dst + i0 * TB), blk + i0 * TB, (i1 - i0) * TB, fb, pol);
                            bulk_g2s(smem_u32(dst + BG * TB + i0 * kScaleTileBytes),
                                     blk + nb * TB + i0 * kScaleTileBytes, (i1 - i0) * kScaleTileBytes, fb, pol);
                        }
                    }
                    ++it;
                    if (++st == nstages) { st = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // Aborted: let copies already issued land before the block can exit.
                const int first = it > nstages ? it - nstages : 0;
                for (int j = first; j < it; ++j)
                    mbar_wait_drain(full0 + 8 * (j % nstages), (j / nstages) & 1, 100000000ull);
                if (nx > 0) mbar_wait_drain(x_full, (nx - 1) & 1, 100000000ull);
            }
        }
        return;
    }

    if (warp == kEpilogueWarp) {
        // ------------------------------------------------------------ epilogue
        // lane takes outputs o = lane + 32 q: q < 8 (gemm: 2 tiles x 128) or q < 4 (swiglu:
        // 128 gate/up pairs). o -> M tile o >> 7, token (o & 127) >> 4, row o & 15.
        constexpr int NQ = SWIGLU ? 4 : 8;
        Segment nat;
        for (int si = 0; si < order.count; ++si) {
            const Segment sg = seg_pick(p, order, si, nat, u1);
            const int b = si & 1;
            named_bar_sync(kBarRedFull + b, kHandoffThreads);
            const float* rb = red + b * kRedFloats;
            float v0[NQ], v1[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int o = lane + 32 * q;
                const int m = SWIGLU ? 0 : (o >> 7), tok = (o & 127) >> 4, row = o & 15;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    s0 += rb[red_index(w, m, tok, row)];
                    if (SWIGLU) s1 += rb[red_index(w, 1, tok, row)];
                }
                v0[q] = s0;
                v1[q] = s1;
            }
            // buffer b is read: hand it back for the run two steps later
            if (si + 2 < order.count) named_bar_arrive(kBarRedFree + b, kHandoffThreads);
            if (flags[0]) continue;
            bool write = segment_complete(p, sg);
            if (!write) {
                // split-K run: publish the partial, take the ticket, reduce if last
                float* ws = a.partials + slot_of(p, sg.s, sg.rp, cta) * kPartialFloats;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    ws[lane + 32 * q] = v0[q];
                    if (SWIGLU) ws[128 + lane + 32 * q] = v1[q];
                }
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = ticket_add(a.tickets + sg.rp) == contributions(p, sg.rp) - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
#pragma unroll
                    for (int q = 0; q < NQ; ++q) v0[q] = v1[q] = 0.f;
                    for (int s = 0; s < p.S; ++s) {
                        const int gs = slab_groups(p, s);
                        const long long r0 = slab_base(p, s) + (long long)sg.rp * gs;
                        const int c_end = cta_of(p, r0 + gs - 1);
                        for (int c = cta_of(p, r0); c <= c_end; ++c) {
                            const float* src = a.partials + slot_of(p, s, sg.rp, c) * kPartialFloats;
#pragma unroll
                            for (int q = 0; q < NQ; ++q) {
                                v0[q] += __ldcg(src + lane + 32 * q);
                                if (SWIGLU) v1[q] += __ldcg(src + 128 + lane + 32 * q);
                            }
                        }
                    }
                    if (lane == 0) a.tickets[sg.rp] = 0;
                    write = true;
                }
            }
            if (write) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const int o = lane + 32 * q;
                    const int m = SWIGLU ? 0 : (o >> 7), tok = (o & 127) >> 4, row = o & 15;
                    const int rt = SWIGLU ? sg.rp : 2 * sg.rp + m;
                    if (tok < T && rt < RT)
                        a.Y[(size_t)tok * p.N + (size_t)rt * kTileRows + row] =
                            SWIGLU ? bf16_bits_rn(silu_mul(v0[q], v1[q])) : bf16_bits_rn(v0[q]);
                }
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

    // The magic constant lives in a register so every decode output is a single LOP3.
    uint32_t magic;
    asm volatile("mov.b32 %0, %1;" : "=r"(magic) : "n"(kBf16Magic));

    // ldmatrix row addresses: lane l serves row (l & 7) of matrix (l >> 3); matrix mi covers
    // K step (mi >> 1) and its half (mi & 1). Absent tokens read the zero row.
    const int lt = lane & 7, mi = lane >> 3;
    const bool lt_valid = lt < T;
    const uint32_t ld_base = lt_valid ? smem_u32(xs + lt * pitch + ((mi >> 1) * 16 + (mi & 1) * 8) * 2)
                                      : smem_u32(zero_row);
    const uint32_t ld_group_step = lt_valid ? 128u : 0u;
    const uint32_t ld_half_step = lt_valid ? 64u : 0u;  // K steps 2,3 are 32 elements further
    // per-lane byte offsets inside a stage's tile area
    const uint32_t code_lane = lane * 16, scale_lane = BG * TB + (lane >> 2) * 4;
    const float* osum_lane = osum + 2 * (lane & 3);

    int st = 0, nx = 0, cur_slab = -1;
    uint32_t phase = 0;
    Segment nat;
    for (int si = 0; si < order.count; ++si) {
        const Segment sg = seg_pick(p, order, si, nat, u1);
        if (sg.s != cur_slab) {
            if (cur_slab >= 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(x_empty);
            }
            mbar_wait(x_full, nx & 1, flags, a.dev_err);
            ++nx;
            cur_slab = sg.s;
            // O[gl][t]: the group MMA chain on the zero-point code, two groups per pass.
            const int gs = slab_groups(p, sg.s);
            const uint32_t az[4] = {kZeroCode, kZeroCode, kZeroCode, kZeroCode};
            for (int gl = warp; gl < gs; gl += 2 * NW) {
                const int gl2 = gl + NW < gs ? gl + NW : gl;
                uint32_t xb[2][8];
                ldsm_x4(ld_base + gl * ld_group_step, xb[0]);
                ldsm_x4(ld_base + gl * ld_group_step + ld_half_step, xb[0] + 4);
                ldsm_x4(ld_base + gl2 * ld_group_step, xb[1]);
                ldsm_x4(ld_base + gl2 * ld_group_step + ld_half_step, xb[1] + 4);
                float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int h = 0; h < 2; ++h) mma_bf16_16816(d[h], az, xb[h][2 * j], xb[h][2 * j + 1]);
                if (lane < 4) {
                    osum[gl * 8 + 2 * lane] = d[0][0];
                    osum[gl * 8 + 2 * lane + 1] = d[0][1];
                    osum[gl2 * 8 + 2 * lane] = d[1][0];
                    osum[gl2 * 8 + 2 * lane + 1] = d[1][1];
                }
            }
            named_bar_sync(kBarConsumers, kConsumerThreads);
        }

        const int rt1 = SWIGLU ? sg.rp : 2 * sg.rp + 1;
        const bool has1 = SWIGLU || rt1 < RT;
        const int slab_g0 = sg.s * GS;
        for (int b = sg.ga / BG; b * BG < sg.gb; ++b) {
            const int i0 = max(sg.ga - b * BG, 0), i1 = min(sg.gb - b * BG, BG);
            const bool ok = mbar_wait(full0 + 8 * st, phase, flags, a.dev_err);
            if (ok) {
                const uint8_t* t0 = stage_mem + st * kStageBytes;
                const int gl0 = b * BG - slab_g0;  // slab-local group of block index 0
                if (i0 == 0 && i1 == BG) {
                    // whole block: groups warp and warp + 8 of both M tiles, K-step-major
                    uint32_t xb[2][8];
                    float2 o[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int gl = gl0 + warp + NW * h;
                        ldsm_x4(ld_base + gl * ld_group_step, xb[h]);
                        ldsm_x4(ld_base + gl * ld_group_step + ld_half_step, xb[h] + 4);
                        o[h] = *reinterpret_cast<const float2*>(osum_lane + gl * 8);
                    }
                    const uint8_t* c0 = t0 + warp * TB + code_lane;
                    const uint8_t* s0 = t0 + scale_lane + warp * kScaleTileBytes;
                    if (has1) {
                        const uint8_t* const code[4] = {c0, c0 + NW * TB, c0 + kTileArea, c0 + kTileArea + NW * TB};
                        const uint8_t* const scale[4] = {s0, s0 + NW * kScaleTileBytes, s0 + kTileArea,
                                                         s0 + kTileArea + NW * kScaleTileBytes};
                        tiles_mma<BITS, 2, 2>(code, scale, xb, o, magic, acc);
                    } else {
                        const uint8_t* const code[2] = {c0, c0 + NW * TB};
                        const uint8_t* const scale[2] = {s0, s0 + NW * kScaleTileBytes};
                        tiles_mma<BITS, 2, 1>(code, scale, xb, o, magic, acc);
                    }
                } else {
                    // part of a block (first or last block of a run): group by group
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int i = warp + NW * h;
                        if (i >= i0 && i < i1) {
                            const int gl = gl0 + i;
                            uint32_t xb[2][8];
                            ldsm_x4(ld_base + gl * ld_group_step, xb[0]);
                            ldsm_x4(ld_base + gl * ld_group_step + ld_half_step, xb[0] + 4);
                            float2 o[2];
                            o[0] = *reinterpret_cast<const float2*>(osum_lane + gl * 8);
                            o[1] = o[0];
                            const uint8_t* c0 = t0 + i * TB + code_lane;
                            const uint8_t* s0 = t0 + scale_lane + i * kScaleTileBytes;
                            if (has1) {
                                const uint8_t* const code[2] = {c0, c0 + kTileArea};
                                const uint8_t* const scale[2] = {s0, s0 + kTileArea};
                                tiles_mma<BITS, 1, 2>(code, scale, xb, o, magic, acc);
                            } else {
                                const uint8_t* const code[1] = {c0};
                                const uint8_t* const scale[1] = {s0};
                                tiles_mma<BITS, 1, 1>(code, scale, xb, o, magic, acc);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
            if (++st == nstages) { st = 0; phase ^= 1; }
        }

        // ------------------------------------------------------------ hand the run over
        const int b = si & 1;
        if (si >= 2) named_bar_sync(kBarRedFree + b, kHandoffThreads);
        float4* r4 = reinterpret_cast<float4*>(red + b * kRedFloats);
        r4[(warp * 2 + 0) * 32 + lane] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        r4[(warp * 2 + 1) * 32 + lane] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
        named_bar_arrive(kBarRedFull + b, kHandoffThreads);
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[m][j] = 0.f;
    }

    if (flags[0] && tid == 0) {
        // Aborted: wait (bounded) for the stage copies that may still be in flight.
        for (int j = 0; j < nstages; ++j) mbar_wait_drain(full0 + 8 * j, 0, 100000000ull);
        for (int j = 0; j < nstages; ++j) mbar_wait_drain(full0 + 8 * j, 1, 100000000ull);
    }
}

}  // namespace nq
