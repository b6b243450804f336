// nq_proj.cuh -- the projection kernel: Y[T,N] = X[T,K] * dequant(W) for T <= 8, 4- or 5-bit
// codes with one fp16 scale per 64-wide K group (or NVFP4 weights), optionally fused into the
// SwiGLU gate/up pair ("NInfer-4090" release post, section "V3 做了什么": small-batch Q4/Q5 projections
// tuned at T=8 for GDN, attention and SwiGLU; "ninfer-ext" README, section
// "与原版 NInfer 的对比": the Q5 K-split MMA path for verify rounds).
//
// Structure: one persistent block per SM with three roles.
//   * Producer warp: its elected lane initialises the mbarriers and streams the block's units
//     with 1-D TMA bulk copies into a ring of shared-memory stages (mbarrier full/empty pairs,
//     L2 evict-first: every weight byte is read exactly once). A stage holds up to 32 groups
//     of each of the two M tiles: one copy of codes and one of scales per tile. It does
//     not wait for the preceding kernel (weights are never written by a kernel that lets its
//     dependents start early); with bf16 operands it holds the stream after the first stage
//     until the activation slab has landed, so the slab's copies do not queue behind a ring.
//   * Consumer warps (kConsumerWarps): they wait for the preceding kernel, stage the X slab
//     of the current K range (fp16 path: cp.async by every thread, then an in-place fp16
//     conversion with a per-token power-of-two range guard; bf16 path: one bulk copy per row)
//     and compute O, the four-MMA chain on the constant zero-point code, for the groups they
//     consume. Warp w then takes K groups w, w + 8, w + 16, w + 24 of every stage, for both
//     16-row tiles of the row pair: a lane decodes its 16 code bytes into A fragments
//     (fp16: 1024 + q, or 1024 + 16 q against X / 16; bf16: 128 + q; exact), loads the B
//     fragment of X with ldmatrix and runs four m16n8k16 MMAs from a zero accumulator: P.
//     The MMA's eight columns are the tokens: token t in column t, or, for up to four tokens
//     (the EVEN instantiations), in column 2t, so that no lane's odd columns hold a token.
//     The warp's eight tiles are issued K-step by K-step so their chains overlap.
//     P - O = sum((q - z) * x) up to fp32 rounding, and exactly 0 where every code equals z
//     (identical MMA inputs). The fp16 scale is applied with one FMA per group.
//   * Two epilogue warps, taking alternate runs: at the end of each (slab, row pair) run the
//     consumers drop their accumulators into one of up to four shared hand-over buffers and
//     carry on. The run's epilogue warp reduces the consumer warps' parts in a fixed order
//     (padded tokens only) and writes Y directly when the run covers its whole pair;
//     otherwise it stores an fp32 partial in the workspace, fences and takes a ticket; the
//     block that takes the last ticket sums all partials of the pair in a fixed order
//     (deterministic split-K, no spinning on other blocks) and writes Y. The block's partial
//     runs are processed first, so split-K settles early and the block ends on a complete run.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "nq_common.cuh"

namespace nq {

constexpr int kMaxGroups = 4;  // projections one grouped launch may carry

struct ProjArgs {
    const uint16_t* X;   // bf16 [T][K]
    const uint8_t* W0;   // packed codes of M tile 0
    const uint8_t* W1;   // M tile 1 (gemm: same matrix, next row tile; swiglu: up matrix)
    const uint8_t* S0;   // packed scales of M tile 0
    const uint8_t* S1;   // packed scales of M tile 1
    uint16_t* Y;         // bf16 [T][N]
    float* partials;     // workspace: slots x kPartialFloats
    int* tickets;        // workspace: one per row pair, zero between calls
    int* dev_err;        // workspace: device error word
    unsigned long long wait_ns;  // bound of every device-side wait
    float gscale = 1.f;  // tensor scale of NVFP4 weights (1 for the integer formats)
    float gscale1 = 1.f; // NVFP4 SwiGLU: tensor scale of the up matrix (M tile 1); gemm: gscale
    // Grouped launch (gemm only): ngroups > 0 projections of the same X, group g owning the
    // global row pairs [gpair[g], gpair[g+1]) with its own packed weight, scales and output
    // (N = gN[g]); W0/W1/S0/S1/Y are then unused. ngroups == 0: one matrix.
    int ngroups = 0;
    int gpair[kMaxGroups + 1];
    int gN[kMaxGroups];
    const uint8_t* gW[kMaxGroups];
    const uint8_t* gS[kMaxGroups];
    uint16_t* gY[kMaxGroups];
    Plan p;              // the real plan (slab geometry, shared memory, grid)
    Plan q;              // work split and split-K bookkeeping: p itself, or the cluster-level
                         // plan of a slab-cluster launch (p.cl > 1)
};

// The matrix a row pair belongs to: its packed codes and scales, output and width, and the
// pair's index inside it.
struct PairLoc {
    const uint8_t* W;
    const uint8_t* S;
    uint16_t* Y;
    int N, RT, rp;
};

__device__ __forceinline__ PairLoc locate_pair(const ProjArgs& a, int rp) {
    if (a.ngroups == 0) return PairLoc{a.W0, a.S0, a.Y, a.p.N, a.p.RT, rp};
    int g = 0;
    while (g + 1 < a.ngroups && rp >= a.gpair[g + 1]) ++g;
    return PairLoc{a.gW[g], a.gS[g], a.gY[g], a.gN[g], a.gN[g] / kTileRows, rp - a.gpair[g]};
}

// Named barriers: 1 = consumers only; 2 + b = run buffer b full (consumers arrive, the
// epilogue warp of that run syncs); 2 + kMaxRed + b = run buffer b free (that epilogue warp
// arrives, consumers sync).
constexpr int kBarConsumers = 1, kBarRedFull = 2, kBarRedFree = 2 + kMaxRed;
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

// A fragment of K step J: fp16 pairs (1024 + q lower-K, 1024 + 16 q upper-K) or bf16 pairs
// (128 + q everywhere).
template <int BITS, bool F16, int J>
__device__ __forceinline__ void decode_step(const uint4& w, uint32_t hb, uint32_t a[4], uint32_t magic) {
    if constexpr (F16) {
        if constexpr (BITS == 4) decode_q4(word_of<J>(w), a, magic);
        else decode_q5<J>(word_of<J>(w), hb, a, magic);
    } else {
        if constexpr (BITS == 4) decode_q4_bf16(word_of<J>(w), a, magic);
        else decode_q5_bf16<J>(word_of<J>(w), hb, a, magic);
    }
}

template <bool F16>
__device__ __forceinline__ void mma_acc(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    if constexpr (F16) mma_f16_16816(d, a, b0, b1); else mma_bf16_16816(d, a, b0, b1);
}

// Which group (B fragments xb[h], O o[h]) and which M tile (acc[m]) tile t of a pass uses:
// GROUPS groups x TILES M tiles, tile t = m * GROUPS + h.
template <int GROUPS>
__device__ __forceinline__ constexpr int group_of(int t) { return t % GROUPS; }
template <int GROUPS>
__device__ __forceinline__ constexpr int mtile_of(int t) { return t / GROUPS; }

// NVFP4, K step J of every tile of a pass: the bare e2m1 values (exact in fp16) go through one
// MMA from a zero accumulator, and the step's partial is added to the accumulator times the
// e4m3 block scales of its two rows, in fp32 (a block of 16 K is one K step). Measured against
// multiplying the scales into the fp16 weights and chaining the four steps: decode shape T = 1
// / 2 / 4 / 8 14.36 / 15.52 / 16.88 / 19.50 -> 12.83 / 14.16 / 15.60 / 19.09 us.
template <int J, int GROUPS, int TILES, bool HALF>
__device__ __forceinline__ void fp4_kstep(const uint4 (&w)[GROUPS * TILES], const uint2 (&sw)[GROUPS * TILES],
                                          const uint32_t (&xb)[GROUPS][8], float (&acc)[2][4]) {
    constexpr int NT = GROUPS * TILES;
    float d[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        // register i of the A fragment: byte i of the lane's word (rows r, r + 8, r, r + 8)
        const uint32_t wj = word_of<J>(w[t]);
        uint32_t a[4];
        a[0] = e2m1x2_to_f16x2(wj);
        a[1] = e2m1x2_to_f16x2(wj >> 8);
        a[2] = e2m1x2_to_f16x2(wj >> 16);
        a[3] = e2m1x2_to_f16x2(wj >> 24);
        mma_zero_16816<true>(d[t], a, xb[group_of<GROUPS>(t)][2 * J], xb[group_of<GROUPS>(t)][2 * J + 1]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        // the e4m3 scales of rows r (low byte) and r + 8 for K step J: bytes 2J, 2J + 1 of the lane's 8
        const uint32_t scj = J < 2 ? (J == 0 ? sw[t].x : sw[t].x >> 16) : (J == 2 ? sw[t].y : sw[t].y >> 16);
        __half2 sh;
        *reinterpret_cast<uint32_t*>(&sh) = e4m3x2_to_f16x2(scj);
        const float2 s = __half22float2(sh);
        const int m = mtile_of<GROUPS>(t);
        acc[m][0] = fmaf(s.x, d[t][0], acc[m][0]);
        acc[m][2] = fmaf(s.y, d[t][2], acc[m][2]);
        if constexpr (!HALF) {  // token columns 2(l%4) + 1: none when tokens sit in even columns
            acc[m][1] = fmaf(s.x, d[t][1], acc[m][1]);
            acc[m][3] = fmaf(s.y, d[t][3], acc[m][3]);
        }
    }
}

// Integer codes, the tiles of a pass: the four K steps of each tile as one MMA chain, then the
// tile's partial P minus its group's zero-point chain O, times the group scale, into acc.
template <int BITS, bool F16, int GROUPS, int TILES, bool HALF>
__device__ __forceinline__ void int_tiles(const uint4 (&w)[GROUPS * TILES], const uint32_t (&hb)[GROUPS * TILES],
                                          const uint2 (&sw)[GROUPS * TILES], const uint32_t (&xb)[GROUPS][8],
                                          const float2 (&o)[GROUPS], uint32_t magic, float (&acc)[2][4]) {
    constexpr int NT = GROUPS * TILES;
    float d[NT][4];
    uint32_t a[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        decode_step<BITS, F16, 0>(w[t], hb[t], a[t], magic);
        mma_zero_16816<F16>(d[t], a[t], xb[group_of<GROUPS>(t)][0], xb[group_of<GROUPS>(t)][1]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        decode_step<BITS, F16, 1>(w[t], hb[t], a[t], magic);
        mma_acc<F16>(d[t], a[t], xb[group_of<GROUPS>(t)][2], xb[group_of<GROUPS>(t)][3]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        decode_step<BITS, F16, 2>(w[t], hb[t], a[t], magic);
        mma_acc<F16>(d[t], a[t], xb[group_of<GROUPS>(t)][4], xb[group_of<GROUPS>(t)][5]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        decode_step<BITS, F16, 3>(w[t], hb[t], a[t], magic);
        mma_acc<F16>(d[t], a[t], xb[group_of<GROUPS>(t)][6], xb[group_of<GROUPS>(t)][7]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int m = mtile_of<GROUPS>(t);
        __half2 sh;
        *reinterpret_cast<uint32_t*>(&sh) = sw[t].x;
        const float2 s = __half22float2(sh);
        const int h = group_of<GROUPS>(t);
        acc[m][0] = fmaf(s.x, d[t][0] - o[h].x, acc[m][0]);
        acc[m][2] = fmaf(s.y, d[t][2] - o[h].x, acc[m][2]);
        if constexpr (!HALF) {  // token columns 2(l%4) + 1: none when tokens sit in even columns
            acc[m][1] = fmaf(s.x, d[t][1] - o[h].y, acc[m][1]);
            acc[m][3] = fmaf(s.y, d[t][3] - o[h].y, acc[m][3]);
        }
    }
}

// GROUPS x TILES tiles in one pass, K-step-major so their accumulator chains overlap. Each
// tile's chain is "K step 0 from a zero accumulator, then K steps 1..3", exactly as for O.
// code[t] / scale[t]: this lane's code bytes / scales of tile t. Integer codes: the tile's
// partial P, minus the zero-point chain O of its group, times the group scale, is added to
// the accumulator. NVFP4: per K step (fp4_kstep).
template <int BITS, bool F16, int GROUPS, int TILES, bool HALF = false>
__device__ __forceinline__ void tiles_mma(const uint8_t* const (&code)[GROUPS * TILES],
                                          const uint8_t* const (&scale)[GROUPS * TILES],
                                          const uint32_t (&xb)[GROUPS][8], const float2 (&o)[GROUPS],
                                          uint32_t magic, float (&acc)[2][4]) {
    constexpr int NT = GROUPS * TILES;
    constexpr bool FP4 = BITS == kFp4;
    uint4 w[NT];
    uint32_t hb[NT];
    uint2 sw[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        w[t] = *reinterpret_cast<const uint4*>(code[t]);
        // high-bit word of the lane: after the tile's 512 nibble bytes, 4 bytes per lane
        hb[t] = BITS == 5 ? *reinterpret_cast<const uint32_t*>(code[t] + 512 - (threadIdx.x & 31) * 12) : 0u;
        if constexpr (FP4)
            sw[t] = *reinterpret_cast<const uint2*>(scale[t]);
        else
            sw[t] = make_uint2(*reinterpret_cast<const uint32_t*>(scale[t]), 0u);
    }
    if constexpr (FP4) {
        fp4_kstep<0, GROUPS, TILES, HALF>(w, sw, xb, acc);
        fp4_kstep<1, GROUPS, TILES, HALF>(w, sw, xb, acc);
        fp4_kstep<2, GROUPS, TILES, HALF>(w, sw, xb, acc);
        fp4_kstep<3, GROUPS, TILES, HALF>(w, sw, xb, acc);
    } else {
        int_tiles<BITS, F16, GROUPS, TILES, HALF>(w, hb, sw, xb, o, magic, acc);
    }
}

// Power-of-two range exponent of one token's X slab from the bits of its max |x| (bf16):
// x * 2^-e has its maximum in [2^14, 2^15), clear of fp16 overflow and far above its
// subnormals; clamped so that 2^e and 2^-e stay normal fp32 numbers.
__device__ __forceinline__ int token_exponent(int max_bits) {
    const int e = ((max_bits >> 7) & 0xFF) - 127 - 14;
    return e < -113 ? -113 : (e > 113 ? 113 : e);
}

// The bf16-operand path keeps fp32's range, but its chains P and O run on offset codes
// (128 + q): with max |x| < 2^100 neither can overflow (|P| < 2^100 * 143 * 64 < 2^114).
// A larger token is scaled by 2^-e, e = (exponent of max |x|) - 99 > 0; otherwise e = 0.
__device__ __forceinline__ int token_exponent_bf16(int max_bits) {
    const int e = ((max_bits >> 7) & 0xFF) - 127 - 99;
    return e < 0 ? 0 : e;
}

// Output element (tile m, token, row) of a run -> its place in the consumers' accumulator
// layout (m16n8 C fragment: lane l holds rows l/4 and l/4+8, tokens 2(l%4) and 2(l%4)+1).
__device__ __forceinline__ int red_index(int w, int m, int tok, int row) {
    const int l = (row & 7) * 4 + (tok >> 1), j = (row >> 3) * 2 + (tok & 1);
    return ((w * 2 + m) * 32 + l) * 4 + j;
}

// EVEN = 0: token t in MMA column t (T <= 8). EVEN = n (1, 2 or 4): at most n tokens, token t
// in column 2t, so that the odd columns of every lane hold no token and need no scaling, and
// the epilogue loops are bounded by n tokens.
template <int BITS, bool SWIGLU, bool F16, int EVEN, bool CLU>
__global__ void __launch_bounds__(kThreads, 1) proj_kernel(const __grid_constant__ ProjArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr bool FP4 = BITS == kFp4;
    constexpr int TB = BITS == 5 ? kQ5TileBytes : kQ4TileBytes;
    constexpr int STB = FP4 ? kFp4ScaleTileBytes : kScaleTileBytes;  // scale bytes per tile
    constexpr int TBS = TB + STB;                     // code + scale bytes per tile
    constexpr int BG = kBlockGroups;                  // groups per block = per stage
    constexpr int kTileArea = BG * TBS;               // one M tile's share of a stage
    constexpr int kStageBytes = 2 * kTileArea;
    constexpr int NW = kConsumerWarps;
    constexpr int kRedFloats = NW * 2 * 128;          // one run buffer
    constexpr int GPW = kGroupsPerWarp;
    static_assert(GPW >= 1 && GPW <= 4, "one to four groups per warp per stage");
    // the zero-point code z in the decode encoding. fp16: 1024 + z for the lower-K registers,
    // 1024 + 16 z for the upper-K registers; bf16: 128 + z everywhere (z = 8 Q4, 16 Q5)
    constexpr uint32_t kZeroLo = F16 ? (BITS == 4 ? 0x64086408u : 0x64106410u) : (BITS == 4 ? 0x43084308u : 0x43104310u);
    constexpr uint32_t kZeroHi = F16 ? (BITS == 4 ? 0x64806480u : 0x65006500u) : kZeroLo;

    // plan fields used in loops, in registers
    const Plan& p = a.p;
    const int T = p.T, G = p.G, GS = p.GS, nstages = p.stages;
    // How the X slab is staged: by every consumer thread (cp.async) for the single-token fp16
    // instantiation, else by one bulk copy per token row, with the weight stream held after its
    // first stage until the rows land. Measured (bulk against cp.async, decode shape): Q4 T = 2
    // 12.7 -> 12.0 us, Q5 verify shape T = 2 10.0 -> 9.25, NVFP4 T = 2 / 4 / 8 14.2 / 15.7 / 19.2
    // -> 13.6 / 14.5 / 17.8; bulk at T = 1 was slower (11.2 -> 11.5). A compile-time choice:
    // the bulk path compiled into the single-token instantiation cost it 0.5-1.7 % (code size).
    constexpr bool kBulkX = !(F16 && EVEN == 1);
    const long long row_tile_codes = (long long)G * TB, row_tile_scales = (long long)G * STB;
    const uint64_t wait_ns = a.wait_ns;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CLU: slab clusters of p.cl blocks; block rank crank takes slab crank of every run of
    // cluster ccta, whose work split is q's. Otherwise q is p and ccta the block.
    const Plan& q = CLU ? a.q : a.p;
    const int crank = CLU ? (int)cluster_rank() : 0;
    const int ccta = CLU ? (int)blockIdx.x / p.cl : (int)blockIdx.x;

    uint8_t* stage_mem = smem;
    uint8_t* xs = smem + nstages * kStageBytes;
    float* osum = reinterpret_cast<float*>(xs + p.x_bytes);  // O[gl][8]
    float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(osum) + p.corr_bytes);  // [2][kRedFloats]
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + p.red_bytes);
    // bars: full[kMaxStages], empty[kMaxStages], x_bar; then flags: [0] abort, [1] stages the
    // producer issued, [2] producer done (both written once the producer stops issuing)
    volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages + 1);
    // per token: max |x| bits of the current slab, then its power-of-two range exponent
    int* xmax = const_cast<int*>(flags) + 8;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
    const uint32_t x_bar = smem_u32(bars + 2 * kMaxStages);  // an activation slab has landed
    // slab clusters: per epilogue warp, "the non-leading ranks' parts have arrived" (rank 0)
    // and "rank 0 has read them" (other ranks); their partial runs land in cbuf of rank 0
    const uint32_t cfull0 = smem_u32(bars + 40), cfree0 = smem_u32(bars + 40 + kEpilogueWarps);
    float* cbuf = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + p.bar_bytes);
    // zero row for ldmatrix lanes of absent tokens: the 16 bytes after the last X row
    const int pitch = x_pitch(GS);
    uint8_t* zero_row = xs + T * pitch;

    const long long u0 = cta_begin(q, ccta), u1 = cta_begin(q, ccta + 1);
    const SegOrder order = seg_order(q, u0, u1);

    if (tid == 0) {
        for (int i = 0; i < nstages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kConsumerWarps);
        }
        mbar_init(x_bar, 1);
        if (CLU) {
            for (int e = 0; e < kEpilogueWarps; ++e) {
                mbar_init(cfull0 + 8 * e, 1);  // rank 0's arrive with the expected bytes
                mbar_init(cfree0 + 8 * e, 1);
            }
        }
        flags[0] = 0;  // abort
        flags[1] = 0;
        flags[2] = 0;
        for (int t = 0; t < 8; ++t) xmax[t] = 0;
        *reinterpret_cast<uint4*>(zero_row) = make_uint4(0, 0, 0, 0);
        mbar_fence_init();
    }
    // Programmatic dependent launch: the next kernel in the stream may be scheduled as SMs
    // free up. The consumers (which read X) and the epilogue warps (which write Y, partial
    // sums and tickets) wait for the preceding kernel to finish (grid_dependency_wait)
    // before they touch global memory. The producer streams the weights at once: no kernel
    // that writes them lets its dependents start early.
    grid_launch_dependents();
    if constexpr (CLU)
        cluster_sync_all();  // every block's barriers are initialised before any remote arrive
    else
        __syncthreads();

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int it = 0, st = 0;
            uint32_t phase = 0;
            bool ok = true;
            Segment nat;
            for (int si = 0; si < order.count && ok; ++si) {
                const Segment v = seg_pick(q, order, si, nat, u1);
                const Segment sg = CLU ? rank_segment(p, v, crank) : v;
                // SwiGLU: tile sg.rp of the gate matrix and of the up matrix; gemm: tiles
                // 2 rp, 2 rp + 1 of the pair's matrix (the second may not exist)
                const PairLoc L = SWIGLU ? PairLoc{a.W0, a.S0, a.Y, p.N, p.RT, sg.rp} : locate_pair(a, sg.rp);
                const int rt0 = SWIGLU ? sg.rp : 2 * L.rp;
                const int rt1 = SWIGLU ? sg.rp : 2 * L.rp + 1;
                const bool has1 = SWIGLU || rt1 < L.RT;
                const uint8_t* w0 = L.W + rt0 * row_tile_codes;
                const uint8_t* w1 = (SWIGLU ? a.W1 : L.W) + rt1 * row_tile_codes;
                const uint8_t* s0 = L.S + rt0 * row_tile_scales;
                const uint8_t* s1 = (SWIGLU ? a.S1 : L.S) + rt1 * row_tile_scales;
                for (int b = sg.ga / BG; sg.ga < sg.gb && b * BG < sg.gb; ++b) {
                    const int i0 = max(sg.ga - b * BG, 0), i1 = min(sg.gb - b * BG, BG);
                    if (!mbar_wait(empty0 + 8 * st, phase ^ 1, flags, a.dev_err, wait_ns)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sb = stage_mem + st * kStageBytes;
                    const uint32_t fb = full0 + 8 * st;
                    const uint32_t per_tile = (i1 - i0) * TBS;
                    mbar_arrive_expect_tx(fb, (has1 ? 2u : 1u) * per_tile);
                    const long long g0 = (long long)b * BG + i0;  // first group of the copy
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        if (m == 1 && !has1) break;
                        uint8_t* dst = sb + m * kTileArea;
                        bulk_g2s(smem_u32(dst + i0 * TB), (m == 0 ? w0 : w1) + g0 * TB, (i1 - i0) * TB, fb, pol);
                        bulk_g2s(smem_u32(dst + BG * TB + i0 * STB), (m == 0 ? s0 : s1) + g0 * STB, (i1 - i0) * STB,
                                 fb, pol);
                    }
                    ++it;
                    // After the first stage, hold the weight stream until a bulk-copied first
                    // activation slab has landed: its copies share this block's copy engine,
                    // and behind a full ring of weight stages they would start the consumers late.
                    if (kBulkX && it == 1 && !mbar_wait(x_bar, 0, flags, a.dev_err, wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (++st == nstages) { st = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // Aborted: let copies already issued land before the block can exit.
                const int first = it > nstages ? it - nstages : 0;
                for (int j = first; j < it; ++j)
                    mbar_wait_drain(full0 + 8 * (j % nstages), (j / nstages) & 1, kDrainNs);
            }
            // Tell the consumers how many stages were issued, for their drain on abort.
            flags[1] = it;
            __threadfence_block();
            flags[2] = 1;
        }
        if constexpr (CLU) cluster_sync_all();  // no block leaves while a peer may address it
        return;
    }

    if (warp >= kEpilogueWarp) {
        // ------------------------------------------------------------ epilogue
        // Two warps take alternate runs, so one run's split-K settle (publish, fence, ticket,
        // fix-up: several L2 round trips under a saturated memory system) overlaps the next.
        // A run has nout outputs o (gemm: M tile, token, row = o / 16TP, (o / 16) % TP,
        // o % 16; swiglu: gate/up pairs, token, row = o / 16, o % 16) over the TP padded
        // tokens only; lane takes o = lane + 32 j.
        const int ew = warp - kEpilogueWarp;
        const int TP = p.TP, nred = p.nred, tp_log = TP == 1 ? 0 : (TP == 2 ? 1 : (TP == 4 ? 2 : 3));
        const int nout = (SWIGLU ? 16 : 32) * TP;
        // Outputs per lane at most: one token (16 or 32 outputs), fp16 path (T <= 2: up to
        // 64), else 8 tokens (256). A compile-time bound keeps the epilogue code small.
        constexpr int kF16TP = NQ_F16_MAX_T <= 1 ? 1 : (NQ_F16_MAX_T <= 2 ? 2 : (NQ_F16_MAX_T <= 4 ? 4 : 8));
        constexpr int kMaxTP = EVEN > 0 ? EVEN : ((F16 && !FP4) ? kF16TP : 8);
        constexpr int JN8 = (SWIGLU ? 16 : 32) * kMaxTP / 32 > 0 ? (SWIGLU ? 16 : 32) * kMaxTP / 32 : 1;
        grid_dependency_wait();  // Y, partial sums and tickets may still be in the preceding kernel's use
        Segment nat;
        int nrun = 0;  // runs this warp has exchanged within the cluster
        for (int si = 0; si < order.count; ++si) {
            const Segment sg = seg_pick(q, order, si, nat, u1);  // cluster-level for CLU
            if ((si & 1) != ew) continue;
            const int b = si % nred;
            named_bar_sync(kBarRedFull + b, kHandoffThreads);
            const float* rb = red + b * kRedFloats;
            float v0[JN8], v1[JN8];
#pragma unroll
            for (int j = 0; j < JN8; ++j) {
                const int o = lane + 32 * j;
                float s0 = 0.f, s1 = 0.f;
                if (o < nout) {
                    const int m = SWIGLU ? 0 : o >> (4 + tp_log), tok = (o >> 4) & (TP - 1), row = o & 15;
                    const float* r0 = rb + red_index(0, m, EVEN > 0 ? 2 * tok : tok, row);
#pragma unroll
                    for (int w = 0; w < NW; ++w) {
                        s0 += r0[w * 256];
                        if (SWIGLU) s1 += r0[w * 256 + 128];
                    }
                }
                v0[j] = s0;
                v1[j] = s1;
            }
            // buffer b is read: hand it back for the run nred steps later
            if (si + nred < order.count) named_bar_arrive(kBarRedFree + b, kHandoffThreads);
            if (flags[0]) continue;
            if constexpr (CLU) {
                // Slab cluster: ranks 1..S-1 store their part of the run into rank 0's buffer
                // for this warp with st.async, which completes the transaction bytes on rank
                // 0's barrier (armed by rank 0 for S-1 parts); rank 0 adds them in rank order
                // and settles the run for the whole cluster. A rank stores its next part only
                // after rank 0 has read the previous one. Layout of a part: [lane][8].
                static_assert(JN8 <= 8 && (SWIGLU ? 2 * JN8 : JN8) <= 8, "one part: 8 values per lane");
                const int S = p.cl;
                const uint32_t fullb = cfull0 + 8 * ew, freeb = cfree0 + 8 * ew;
                constexpr uint32_t kPartBytes = 32 * 8 * 4;
                if (crank != 0) {
                    if (nrun > 0 && !mbar_wait_cluster(freeb, (nrun - 1) & 1, flags, a.dev_err, wait_ns)) continue;
                    float w[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) w[j] = 0.f;
#pragma unroll
                    for (int j = 0; j < JN8; ++j) {
                        w[j] = v0[j];
                        if (SWIGLU) w[JN8 + j] = v1[j];
                    }
                    const uint32_t dst = cluster_map(
                        smem_u32(cbuf + (ew * (S - 1) + crank - 1) * kPartialFloats + lane * 8), 0);
                    const uint32_t rbar = cluster_map(fullb, 0);
                    cluster_store_async_v4(dst, w[0], w[1], w[2], w[3], rbar);
                    cluster_store_async_v4(dst + 16, w[4], w[5], w[6], w[7], rbar);
                    ++nrun;
                    continue;
                }
                if (lane == 0) mbar_arrive_expect_tx(fullb, (uint32_t)(S - 1) * kPartBytes);
                if (!mbar_wait_cluster(fullb, nrun & 1, flags, a.dev_err, wait_ns)) continue;
                for (int r = 1; r < S; ++r) {
                    const float* src = cbuf + (ew * (S - 1) + r - 1) * kPartialFloats + lane * 8;
#pragma unroll
                    for (int j = 0; j < JN8; ++j) {
                        v0[j] += src[j];
                        if (SWIGLU) v1[j] += src[JN8 + j];
                    }
                }
                __syncwarp();
                if (lane == 0)
                    for (int r = 1; r < S; ++r) mbar_arrive_remote(cluster_map(freeb, r));
                ++nrun;
            }
            bool write = segment_complete(q, sg);
            if (!write) {
                // split-K run: publish the partial, take the ticket, reduce if last
                float* ws = a.partials + slot_of(q, sg.s, sg.rp, ccta) * kPartialFloats;
#pragma unroll
                for (int j = 0; j < JN8; ++j) {
                    const int o = lane + 32 * j;
                    if (o < nout) {
                        ws[o] = v0[j];
                        if (SWIGLU) ws[128 + o] = v1[j];
                    }
                }
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    fence_acq_rel_gpu();  // the warp's partial stores before the ticket
                    last = ticket_add(a.tickets + sg.rp) == contributions(q, sg.rp) - 1;
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
#pragma unroll
                    for (int j = 0; j < JN8; ++j) v0[j] = v1[j] = 0.f;
                    // Every contribution of the pair, summed in fixed (slab, block) order.
                    auto sum_in_order = [&]() {
                        for (int s = 0; s < q.S; ++s) {
                            const int gs = slab_groups(q, s);
                            const long long r0 = slab_base(q, s) + (long long)sg.rp * gs;
                            const int c_end = cta_of(q, r0 + gs - 1);
                            for (int c = cta_of(q, r0); c <= c_end; ++c) {
                                const float* src = a.partials + slot_of(q, s, sg.rp, c) * kPartialFloats;
#pragma unroll
                                for (int j = 0; j < JN8; ++j) {
                                    const int o = lane + 32 * j;
                                    if (o < nout) {
                                        v0[j] += __ldcg(src + o);
                                        if (SWIGLU) v1[j] += __ldcg(src + 128 + o);
                                    }
                                }
                            }
                        }
                    };
                    if constexpr (F16) {
                        sum_in_order();  // one slab: two or three contributions
                    } else {
                        // Several slabs: the loads go out kBatch contributions at a time (same
                        // order), so their L2 round trips overlap instead of queueing.
                        constexpr int kFix = 16, kBatch = 4, JN = SWIGLU ? 4 : 8;
                        int slots[kFix];
                        int nc = 0;
                        for (int s = 0; s < q.S; ++s) {
                            const int gs = slab_groups(q, s);
                            const long long r0 = slab_base(q, s) + (long long)sg.rp * gs;
                            const int c_end = cta_of(q, r0 + gs - 1);
                            for (int c = cta_of(q, r0); c <= c_end; ++c) {
                                if (nc < kFix) slots[nc] = (int)slot_of(q, s, sg.rp, c);
                                ++nc;
                            }
                        }
                        if (nc > kFix) {
                            sum_in_order();
                        } else {
                            for (int k0 = 0; k0 < nc; k0 += kBatch) {
                                float t0[kBatch][JN], t1[kBatch][JN];
#pragma unroll
                                for (int u = 0; u < kBatch; ++u) {
                                    const float* src = a.partials + (size_t)slots[k0 + u < nc ? k0 + u : k0] * kPartialFloats;
#pragma unroll
                                    for (int j = 0; j < JN; ++j) {
                                        const int o = lane + 32 * j;
                                        t0[u][j] = t1[u][j] = 0.f;
                                        if (k0 + u < nc && o < nout) {
                                            t0[u][j] = __ldcg(src + o);
                                            if (SWIGLU) t1[u][j] = __ldcg(src + 128 + o);
                                        }
                                    }
                                }
#pragma unroll
                                for (int u = 0; u < kBatch; ++u)
#pragma unroll
                                    for (int j = 0; j < JN; ++j)
                                        if (k0 + u < nc) {
                                            v0[j] += t0[u][j];
                                            v1[j] += t1[u][j];
                                        }
                            }
                        }
                    }
                    if (lane == 0) a.tickets[sg.rp] = 0;
                    write = true;
                }
            }
            if (write) {
                const PairLoc L = SWIGLU ? PairLoc{a.W0, a.S0, a.Y, p.N, p.RT, sg.rp} : locate_pair(a, sg.rp);
#pragma unroll
                for (int j = 0; j < JN8; ++j) {
                    const int o = lane + 32 * j;
                    const int m = SWIGLU ? 0 : o >> (4 + tp_log), tok = (o >> 4) & (TP - 1), row = o & 15;
                    const int rt = SWIGLU ? sg.rp : 2 * L.rp + m;
                    if (o < nout && tok < T && rt < L.RT)
                        L.Y[(size_t)tok * L.N + (size_t)rt * kTileRows + row] =
                            SWIGLU ? bf16_bits_rn(silu_mul(v0[j], v1[j])) : bf16_bits_rn(v0[j]);
                }
            }
        }
        if constexpr (CLU) cluster_sync_all();
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
    asm volatile("mov.b32 %0, %1;" : "=r"(magic) : "n"(F16 ? kF16Magic : kBf16Magic));

    // ldmatrix row addresses: lane l serves row (l & 7) of matrix (l >> 3), i.e. MMA column
    // l & 7; matrix mi covers K step (mi >> 1) and its half (mi & 1). Columns without a token
    // (past T; with EVEN, the odd ones) read the zero row.
    const int lt = lane & 7, mi = lane >> 3;
    const int ltok = EVEN > 0 ? lt >> 1 : lt;
    const bool lt_valid = (EVEN == 0 || (lt & 1) == 0) && ltok < T;
    const uint32_t ld_base = lt_valid ? smem_u32(xs + ltok * pitch + ((mi >> 1) * 16 + (mi & 1) * 8) * 2)
                                      : smem_u32(zero_row);
    const uint32_t ld_group_step = lt_valid ? 128u : 0u;
    const uint32_t ld_half_step = lt_valid ? 64u : 0u;  // K steps 2,3 are 32 elements further
    // per-lane byte offsets inside a stage's tile area
    const uint32_t code_lane = lane * 16, scale_lane = BG * TB + (lane >> 2) * (FP4 ? 8 : 4);
    const float* osum_lane = osum + 2 * (lane & 3);

    int st = 0, cur_slab = -1, nx = 0, nx_issued = 0;
    uint32_t phase = 0;
    float tok_scale0 = 1.f, tok_scale1 = 1.f;
    Segment nat;
    for (int si = 0; si < order.count; ++si) {
        const Segment v = seg_pick(q, order, si, nat, u1);
        const Segment sg = CLU ? rank_segment(p, v, crank) : v;
        if (sg.s != cur_slab) {
            if (cur_slab >= 0)
                named_bar_sync(kBarConsumers, kConsumerThreads);  // all done with the old slab
            else
                grid_dependency_wait();  // X may be the preceding kernel's output
            cur_slab = sg.s;
            const int gs = slab_groups(p, sg.s);
            const int chunks = gs * 8;  // 16-byte chunks per token row
            // The X slab into shared memory. One token row (the single-token instantiation):
            // 16-byte copies by every consumer thread (LSU path, off the weight stream's copy
            // engine). More rows: one bulk copy per row, since the LSU path stages through the
            // L1 left beside this block's shared memory and would take several round trips.
            const uint16_t* xg = a.X + (size_t)sg.s * GS * kGroup;
            if constexpr (!kBulkX) {
                for (int t = 0; t < T; ++t)
                    for (int c = tid; c < chunks; c += kConsumerThreads)
                        cp_async16(smem_u32(xs + t * pitch + c * 16), xg + (size_t)t * p.K + c * 8);
                cp_async_wait_all();  // each thread's own chunks; the range pass below reads only those
            } else {
                if (tid == 0) {
                    // The previous slab's copies have landed (every consumer waited for them,
                    // unless the block aborted: then wait here, bounded), so phases never
                    // overlap; after an abort no new slab is fetched.
                    if (nx_issued > 0) mbar_wait_drain(x_bar, (nx_issued - 1) & 1, kDrainNs);
                    if (!flags[0]) {
                        const uint32_t row_bytes = gs * 128;
                        mbar_arrive_expect_tx(x_bar, row_bytes * T);
                        for (int t = 0; t < T; ++t)
                            bulk_g2s_plain(smem_u32(xs + t * pitch), xg + (size_t)t * p.K, row_bytes, x_bar);
                        ++nx_issued;
                    }
                }
                mbar_wait(x_bar, nx & 1, flags, a.dev_err, wait_ns);
                ++nx;
            }
            // Per token, max |x| over the slab (bit patterns compare like magnitudes), then the
            // operand conversion and O[gl][t], the group MMA chain on the zero-point code. The
            // fp16 path always needs the maximum. The bf16 path needs it only when some |x|
            // reaches 2^100 (bits 0x7180): the O pass, which loads every group of the slab
            // once across the warps, also tests its fragments; a barrier OR-reduction decides,
            // and only then do the max pass, the rescale and a second O pass run.
            if (tid < 8) xmax[tid] = 0;
            if constexpr (F16) named_bar_sync(kBarConsumers, kConsumerThreads);
            bool need_max = F16;
            for (int rep = 0;; ++rep) {
                if (need_max) {
                    for (int t = 0; t < T; ++t) {
                        uint32_t mx = 0;
                        for (int c = tid; c < chunks; c += kConsumerThreads) {
                            const uint4 v = *reinterpret_cast<const uint4*>(xs + t * pitch + c * 16);
                            const uint32_t m = max(max(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                                   max(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
                            mx = max(mx, max(m & 0xFFFFu, m >> 16));
                        }
                        mx = __reduce_max_sync(0xffffffffu, mx);
                        if (lane == 0) atomicMax(xmax + t, (int)mx);
                    }
                    named_bar_sync(kBarConsumers, kConsumerThreads);
                    if constexpr (F16) {
                        // X slab bf16 -> fp16 in place, times 2^-e (token_exponent); the upper-K
                        // half of every 16-wide K step is also divided by 16 (see decode_q4).
                        // Both exact.
                        for (int t = 0; t < T; ++t) {
                            const int e = token_exponent(xmax[t]);
                            const float lo_scale = __int_as_float((127 - e) << 23);
                            const float hi_scale = FP4 ? lo_scale : lo_scale * 0.0625f;
                            for (int c = tid; c < chunks; c += kConsumerThreads) {
                                uint4* q = reinterpret_cast<uint4*>(xs + t * pitch + c * 16);
                                const uint4 v = *q;
                                const float sc = (c & 1) ? hi_scale : lo_scale;
                                uint4 o;
                                uint32_t* ov = reinterpret_cast<uint32_t*>(&o);
                                const uint32_t* iv = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const __half2 h2 = __floats2half2_rn(__uint_as_float(iv[i] << 16) * sc,
                                                                         __uint_as_float(iv[i] & 0xFFFF0000u) * sc);
                                    ov[i] = *reinterpret_cast<const uint32_t*>(&h2);
                                }
                                *q = o;
                            }
                        }
                    } else {
                        // bf16 operands: only a token too large for the offset chains is rescaled.
                        for (int t = 0; t < T; ++t) {
                            const int e = token_exponent_bf16(xmax[t]);
                            if (e == 0) continue;
                            const float sc = __int_as_float((127 - e) << 23);
                            for (int c = tid; c < chunks; c += kConsumerThreads) {
                                uint4* q = reinterpret_cast<uint4*>(xs + t * pitch + c * 16);
                                uint4 v = *q;
                                uint32_t* iv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(iv[i] << 16) * sc,
                                                                                    __uint_as_float(iv[i] & 0xFFFF0000u) * sc);
                                    iv[i] = *reinterpret_cast<const uint32_t*>(&b2);
                                }
                                *q = v;
                            }
                        }
                    }
                    named_bar_sync(kBarConsumers, kConsumerThreads);
                }
                // O[gl][t]: a warp consumes only the groups gl = warp (mod NW) of the slab
                // (blocks start on multiples of NW), so it computes exactly those, four chains
                // per pass, and only it reads them back. big: some half of a fragment has
                // |x| >= 2^100 (a 15-bit magnitude m >= 0x7180 carries into bit 15 of
                // m + 0x0E80, and no further).
                uint32_t big = 0;
                const uint32_t az[4] = {kZeroLo, kZeroLo, kZeroHi, kZeroHi};
                if constexpr (F16 && EVEN == 1 && !FP4) {
                    // One token: the chain's column for one group does not depend on the other
                    // columns (outputs bit-identical), so eight of the warp's groups share a chain,
                    // column c taking group warp + NW (c + 8 j); the other columns of O[g] are zero.
                    // Against four single-group chains per pass: K = 17408 16.25 -> 15.98 us, Q5
                    // K = 5120 8.30 -> 8.26, Q4 decode shape unchanged.
                    for (int j = 0; warp + 8 * NW * j < gs; ++j) {
                        const int gc0 = warp + NW * (lt + 8 * j);
                        const int gc = gc0 < gs ? gc0 : warp;
                        const uint32_t la = smem_u32(xs) + gc * 128u + ((mi >> 1) * 16 + (mi & 1) * 8) * 2;
                        uint32_t xb[8];
                        ldsm_x4(la, xb);
                        ldsm_x4(la + 64u, xb + 4);
                        float d[4];
                        mma_zero_16816<true>(d, az, xb[0], xb[1]);
                        mma_acc<true>(d, az, xb[2], xb[3]);
                        mma_acc<true>(d, az, xb[4], xb[5]);
                        mma_acc<true>(d, az, xb[6], xb[7]);
                        if (lane < 4) {  // columns 2 lane, 2 lane + 1
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int g = warp + NW * (2 * lane + h + 8 * j);
                                if (g < gs) {
                                    float4* row = reinterpret_cast<float4*>(osum + g * 8);
                                    row[0] = make_float4(d[h], 0.f, 0.f, 0.f);
                                    row[1] = make_float4(0.f, 0.f, 0.f, 0.f);
                                }
                            }
                        }
                    }
                }
                for (int gl = warp; !FP4 && !(F16 && EVEN == 1) && gl < gs; gl += 4 * NW) {  // NVFP4: no zero point
                    int g[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) g[c] = gl + c * NW < gs ? gl + c * NW : gl;
                    uint32_t xb[4][8];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        ldsm_x4(ld_base + g[c] * ld_group_step, xb[c]);
                        ldsm_x4(ld_base + g[c] * ld_group_step + ld_half_step, xb[c] + 4);
                    }
                    if constexpr (!F16) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int i = 0; i < 8; ++i) big |= (xb[c][i] & 0x7FFF7FFFu) + 0x0E800E80u;
                    }
                    float d[4][4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) mma_zero_16816<F16>(d[c], az, xb[c][0], xb[c][1]);
#pragma unroll
                    for (int j = 1; j < 4; ++j)
#pragma unroll
                        for (int c = 0; c < 4; ++c) mma_acc<F16>(d[c], az, xb[c][2 * j], xb[c][2 * j + 1]);
                    if (lane < 4) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<float2*>(osum + g[c] * 8 + 2 * lane) = make_float2(d[c][0], d[c][1]);
                    }
                }
                if (F16 || rep > 0) break;
                need_max = named_bar_or(kBarConsumers, kConsumerThreads, (big & 0x80008000u) != 0);
                if (!need_max) break;
            }
            __syncwarp();
            // 2^e of the lane's two token columns (from the max bits), applied at the hand-over
            {
                const int m0 = xmax[EVEN > 0 ? (lane & 3) : 2 * (lane & 3)];
                const int m1 = EVEN > 0 ? m0 : xmax[2 * (lane & 3) + 1];
                const int e0 = F16 ? token_exponent(m0) : token_exponent_bf16(m0);
                const int e1 = F16 ? token_exponent(m1) : token_exponent_bf16(m1);
                tok_scale0 = __int_as_float((127 + e0) << 23);
                tok_scale1 = __int_as_float((127 + e1) << 23);
            }
        }

        // Both M tiles always run: when the pair's second row tile does not exist (odd tile
        // count, last pair) its chains run on whatever the stage holds there and the result is
        // never stored (the epilogue drops rows past N). One code path keeps the loop small
        // enough for the instruction cache.
        const int slab_g0 = sg.s * GS;
        for (int b = sg.ga / BG; sg.ga < sg.gb && b * BG < sg.gb; ++b) {
            const int i0 = max(sg.ga - b * BG, 0), i1 = min(sg.gb - b * BG, BG);
            const bool ok = mbar_wait(full0 + 8 * st, phase, flags, a.dev_err, wait_ns);
            if (ok) {
                const uint8_t* t0 = stage_mem + st * kStageBytes;
                const int gl0 = b * BG - slab_g0;  // slab-local group of block index 0
                // this warp's first group of the block: X fragment address and O pointer
                const uint32_t la0 = ld_base + (gl0 + warp) * ld_group_step;
                const float* o0 = osum_lane + (gl0 + warp) * 8;
                if (i0 == 0 && i1 == BG) {
                    // whole block: this warp's GPW groups of both M tiles, K-step-major
                    uint32_t xb[GPW][8];
                    float2 o[GPW];
#pragma unroll
                    for (int h = 0; h < GPW; ++h) {
                        const uint32_t la = la0 + (NW * h) * ld_group_step;
                        ldsm_x4(la, xb[h]);
                        ldsm_x4(la + ld_half_step, xb[h] + 4);
                        o[h] = *reinterpret_cast<const float2*>(o0 + 8 * NW * h);
                    }
                    const uint8_t* c0 = t0 + warp * TB + code_lane;
                    const uint8_t* s0 = t0 + scale_lane + warp * STB;
                    const uint8_t* code[2 * GPW];
                    const uint8_t* scale[2 * GPW];
#pragma unroll
                    for (int t = 0; t < 2 * GPW; ++t) {
                        const int m = t / GPW, h = t % GPW;
                        code[t] = c0 + m * kTileArea + NW * h * TB;
                        scale[t] = s0 + m * kTileArea + NW * h * STB;
                    }
                    tiles_mma<BITS, F16, GPW, 2, (EVEN > 0)>(code, scale, xb, o, magic, acc);
                } else if (i0 == 0 && i1 == BG / 2) {
                    // the first half of a block (the 16-group tail of a row whose group count
                    // is 16 mod 32, e.g. K = 5120): groups warp and warp + NW, unrolled
                    constexpr int H = GPW / 2;
                    uint32_t xb[H][8];
                    float2 o[H];
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const uint32_t la = la0 + (NW * h) * ld_group_step;
                        ldsm_x4(la, xb[h]);
                        ldsm_x4(la + ld_half_step, xb[h] + 4);
                        o[h] = *reinterpret_cast<const float2*>(o0 + 8 * NW * h);
                    }
                    const uint8_t* c0 = t0 + warp * TB + code_lane;
                    const uint8_t* s0 = t0 + scale_lane + warp * STB;
                    const uint8_t* code[2 * H];
                    const uint8_t* scale[2 * H];
#pragma unroll
                    for (int t = 0; t < 2 * H; ++t) {
                        const int m = t / H, h = t % H;
                        code[t] = c0 + m * kTileArea + NW * h * TB;
                        scale[t] = s0 + m * kTileArea + NW * h * STB;
                    }
                    tiles_mma<BITS, F16, H, 2, (EVEN > 0)>(code, scale, xb, o, magic, acc);
                } else {
                    // part of a block (first or last block of a run): group by group, in a
                    // loop that is not unrolled (rare, and it keeps the code small)
#pragma unroll 1
                    for (int h = 0; h < GPW; ++h) {
                        const int i = warp + NW * h;
                        if (i >= i0 && i < i1) {
                            uint32_t xb[1][8];
                            const uint32_t la = la0 + (NW * h) * ld_group_step;
                            ldsm_x4(la, xb[0]);
                            ldsm_x4(la + ld_half_step, xb[0] + 4);
                            const float2 o[1] = {*reinterpret_cast<const float2*>(o0 + 8 * NW * h)};
                            const uint8_t* c0 = t0 + i * TB + code_lane;
                            const uint8_t* s0 = t0 + scale_lane + i * STB;
                            const uint8_t* const code[2] = {c0, c0 + kTileArea};
                            const uint8_t* const scale[2] = {s0, s0 + kTileArea};
                            tiles_mma<BITS, F16, 1, 2, (EVEN > 0)>(code, scale, xb, o, magic, acc);
                        }
                    }
                }
            }
            __syncwarp();
            mbar_arrive_if(empty0 + 8 * st, lane == 0);
            if (++st == nstages) { st = 0; phase ^= 1; }
        }

        // ------------------------------------------------------------ hand the run over
        const int b = si % p.nred;
        if (si >= p.nred) named_bar_sync(kBarRedFree + b, kHandoffThreads);
        float4* r4 = reinterpret_cast<float4*>(red + b * kRedFloats);
        {
            // NVFP4: the tensor scale of M tile m's matrix (for SwiGLU, gate or up) joins the
            // token scales (a power of two: exact)
            const float g0 = FP4 ? a.gscale : 1.f, g1 = FP4 ? a.gscale1 : 1.f;
            const float a0 = tok_scale0 * g0, a1 = tok_scale1 * g0, b0 = tok_scale0 * g1, b1 = tok_scale1 * g1;
            r4[(warp * 2 + 0) * 32 + lane] = make_float4(acc[0][0] * a0, acc[0][1] * a1, acc[0][2] * a0, acc[0][3] * a1);
            r4[(warp * 2 + 1) * 32 + lane] = make_float4(acc[1][0] * b0, acc[1][1] * b1, acc[1][2] * b0, acc[1][3] * b1);
        }
        named_bar_arrive(kBarRedFull + b, kHandoffThreads);
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[m][j] = 0.f;
    }

    if (flags[0] && tid == 0) {
        // Aborted: the consumers stopped waiting for their stages, so copies may still be in
        // flight. Once the producer has stopped (bounded wait for its flag), wait (bounded)
        // for the last copy issued into each stage -- a stage's phases complete in order --
        // and for the last activation slab.
        const uint64_t t0 = global_timer_ns();
        while (!flags[2] && global_timer_ns() - t0 < 2 * kDrainNs) {
        }
        const int issued = flags[1];
        for (int j = issued > nstages ? issued - nstages : 0; j < issued; ++j)
            mbar_wait_drain(full0 + 8 * (j % nstages), (j / nstages) & 1, kDrainNs);
        if (nx_issued > 0) mbar_wait_drain(x_bar, (nx_issued - 1) & 1, kDrainNs);
    }
    if constexpr (CLU) cluster_sync_all();
}

}  // namespace nq
