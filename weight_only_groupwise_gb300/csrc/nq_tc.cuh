// nq_tc.cuh -- the large-batch projection kernel: Y[T,N] = X[T,K] * dequant(W) for
// 8 < T <= 64 tokens (several concurrent requests' speculative-verify rows: "ninfer-ext"
// README, section "与原版 NInfer 的对比", C = 1..8 requests; "NInfer-4090" post, section
// "实测数据", C2/C4/C8), 4- or 5-bit codes with one fp16 scale per 64-wide K group or NVFP4
// weights, on the fifth-generation tensor cores (tcgen05) so that the weights stream from HBM
// once whatever T. A SwiGLU block is two launches (the output-mode template argument): the
// gate projection writes fp32 G, the up projection writes bf16 silu(G) * U.
//
// One block per (128-row block, K piece), D + E + 3 warps (D decoders: 8, or 16 for NVFP4 with
// TP <= 32; E epilogue warps: 4, or 8 for 4/5-bit codes at TP = 64). Work moves between the
// warp roles in stages of BG 64-wide K groups (six for TP <= 32 padded tokens, four for
// TP = 64: the TMEM budget), one hand-off per stage:
//   * warp 0, one lane -- producer: per stage three 3-D TMA copies: the codes and the scales of
//     the eight 16-row tiles (tiles and groups past the matrix read as zeros), and the stage's
//     activation chunk, one [TP][64] block per group in the tensor core's K-major
//     128-byte-swizzled layout, tokens past T filled with zeros by the copy. A ring of
//     shared-memory stages (1024-byte aligned), mbarriers.
//   * warps 1..D -- decoders: warp w owns one 16-row tile, TMEM lanes 32 (w % 4) + 16 h .. + 15
//     (h = 0 for warps 1..4, 1 for 5..8, and again for 9..16, which take the odd groups of
//     each stage when D = 16). A lane decodes its fragment words of a group into
//     bf16 (q - z) 2^-12, exact, and stores all four K steps with one tcgen05.st.16x128b.x8,
//     which places the mma.sync A-fragment registers of lane t at TMEM lanes t/4, t/4 + 8 and
//     columns 8 j + t%4, 8 j + 4 + t%4: K in natural order, one row per TMEM lane. An A buffer
//     holds a stage (32 columns a group); two alternate. Groups are decoded in pairs (D = 8)
//     or one by one (D = 16), each into registers of its own, so that they decode while the
//     stores of the groups before them complete.
//   * warps D + 1, D + 2 -- MMA issuers, alternate P buffers (the whole warp runs the loop, one
//     elected lane issues): per group, four tcgen05.mma.kind::f16 (M = 128, N = TP, K = 16;
//     A from TMEM, B = the activation chunk through a shared-memory descriptor; D in TMEM,
//     fp32, a fresh accumulator per group: P = 2^-12 sum over the group of (q - z) x); per P
//     buffer (two or three groups) a tcgen05.commit publishes their P, per stage each issuer's
//     commits free the A buffer and the shared-memory stage.
//   * warps D + 3 .. D + E + 2 -- epilogue: thread = row (TMEM lane) and E / 4 token ranges;
//     per group it loads P (tcgen05.ld) and adds 2^12 s[row, g] * P[t] to its fp32
//     accumulators acc[t] of its tokens. At the end it stores bf16 Y,
//     or, when K is split across blocks, an fp32 partial; the last block of a row block
//     (ticket) adds the partials in fixed order and stores Y.
// The 2^-12 in the decoded weights keeps every group partial finite for any finite bf16
// activation: |q - z| 2^-12 <= 2^-8 and |x| < 2^128, so 64 products stay below 2^126 (fp32
// overflows at 2^128); 2^12 s is exact in fp32, so the result is the unscaled one. No range
// pass over the activations is needed.
// Every wait is bounded (the abort protocol of the small-batch kernel); TMEM is allocated and
// freed by warp 0, after the issuers have waited for their last MMAs. With one block per SM the
// kernel takes all 512 TMEM columns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "nq_common.cuh"

namespace nq {

constexpr int kTcRows = 128;                      // rows per block = MMA M
constexpr int kTcTiles = kTcRows / kTileRows;     // 16-row tiles per block
constexpr int kTcMaxStages = 8;
constexpr int kTcPair = 2;                        // groups per decode step and per P buffer
constexpr int kTcA = 2;                           // A buffers in TMEM (a stage: 32 columns a group)
constexpr int kTcCols = 512;                      // TMEM columns: A buffers, then P buffers
constexpr int kTcMaxP = 8;
constexpr int kTcScaleExp = 12;                   // decoded 4/5-bit weights carry 2^-12
constexpr int kTcFp4ScaleExp = 20;                // decoded NVFP4 weights carry 2^-20
// Decoder warps: one per 16-row tile; two (each every other group of a stage) for NVFP4 with
// TP <= 32, whose decode (e2m1 x e4m3 to fp16, then bf16) is the longest, and for 5-bit codes
// at TP = 16. Measured at T = 16: NVFP4 on the decode shape 26.7 -> 24.5 us, Q5 on the verify
// shape 11.7 -> 11.4 us; slower for Q4 (16.0 -> 16.5: it loses the one-store pairs) and for
// Q5 at TP = 32 (13.0 -> 13.2); at TP = 64 the epilogue accumulators need the registers of the
// smaller block.
NQ_HD constexpr int tc_decoders(int bits, int TP) {
    return (bits == kFp4 && TP <= 32) || (bits == 5 && TP == 16) ? 16 : 8;
}
// Epilogue warps: one per TMEM lane quarter (all the tokens of its 32 rows), or two per quarter
// (each half the tokens) for 4/5-bit codes at TP = 64, where one warp's 64 accumulators and
// loads set the pace. Measured at T = 64 (with two issuers): decode shape 22.3 -> 21.7 us,
// 5120 x 6144 Q5 15.9 -> 15.1, down projection 28.6 -> 27.6; NVFP4 gains nothing and keeps four.
NQ_HD constexpr int tc_epilogues(int bits, int TP) { return TP == 64 && bits != kFp4 ? 8 : 4; }
// MMA issuers: two warps on different SM sub-partitions take alternate P steps. A single
// issuer slowed the other warps of its sub-partition (traced: its decoder and epilogue warps
// finished each hand-off about 0.35 us after the others), and every hand-off waits for the
// slowest TMEM lane quarter. Measured, one issuer -> two, T = 16 / 32: decode shape Q4 16.6 /
// 18.9 -> 16.0 / 18.6 us, down projection 20.2 / 23.1 -> 19.6 / 22.6, NVFP4 23.7 / 26.0 ->
// 23.3 / 25.5 (T = 64: 30.4 -> 29.8); 5120 x 6144 Q5 unchanged. Three issuers won on some
// shapes and lost on others.
constexpr int kTcIssuers = 2;
NQ_HD constexpr int tc_threads(int bits, int TP) {
    return (1 + tc_decoders(bits, TP) + kTcIssuers + tc_epilogues(bits, TP)) * 32;
}
constexpr int kTcMinT = 9, kTcMaxT = 64;
// What the epilogue writes for (token t, row n) from the finished fp32 value v: bf16 Y = v;
// fp32 G = v (a SwiGLU gate projection); bf16 Y = silu(G) * v (the up projection of the same
// SwiGLU block, G written by the preceding launch). A template argument of the kernel: the
// final stores are unrolled over the tokens, and a run-time choice there would multiply that
// code (measured +5 % at TP = 16 and +16 % at TP = 64 on plain projections).
constexpr int kTcOutY = 0, kTcOutGate = 1, kTcOutSwiglu = 2;

// 64-wide K groups per pipeline stage (one hand-off between the warp roles). Six while the P
// buffers of two groups fit beside two six-group A buffers (2 x 192 + 2 x 2 TP <= 512 TMEM
// columns: TP <= 32), else four, which leaves the 64-token kernel its four stages.
NQ_HD constexpr int tc_stage_groups(int TP) { return TP <= 32 ? 6 : 4; }
// Shared-memory bytes of one stage: codes and scales of kTcTiles tiles x BG groups, then the
// activation chunk (BG * 64 K x TP tokens, bf16).
NQ_HD constexpr int tc_weight_bytes(int bits, int TP) {
    return kTcTiles * tc_stage_groups(TP) * (code_tile_bytes(bits) + scale_tile_bytes(bits));
}
NQ_HD constexpr int tc_x_bytes(int TP) { return TP * tc_stage_groups(TP) * kGroup * 2; }
// The weights of a stage padded to 1024 bytes: the activation chunk after them starts on a
// 1024-byte boundary (the swizzle atom).
NQ_HD constexpr int tc_weight_region(int bits, int TP) { return (tc_weight_bytes(bits, TP) + 1023) / 1024 * 1024; }
NQ_HD constexpr int tc_stage_bytes(int bits, int TP) { return tc_weight_region(bits, TP) + tc_x_bytes(TP); }
// Alignment of the stages to 1024 bytes (the swizzle atom), then barriers and flags after them.
NQ_HD constexpr int tc_extra_bytes(int) { return 2048; }
NQ_HD constexpr int tc_stages(int bits, int TP) {
    int s = (kSmemLimit - tc_extra_bytes(TP)) / tc_stage_bytes(bits, TP);
    return s > kTcMaxStages ? kTcMaxStages : s;
}
NQ_HD constexpr int tc_tpad(int T) { return T <= 16 ? 16 : (T <= 32 ? 32 : 64); }

// Work split of a large-batch call: RB row blocks of 128 rows, each K cut into KS pieces so
// that RB * KS blocks about fill the SMs.
struct TcPlan {
    int T, TP, K, N, G, RT, RB, KS, P, stages, smem_bytes;
};

NQ_HD bool make_tc_plan(int bits, int T, int K, int N, int num_sms, TcPlan& p) {
    p.T = T;
    p.TP = tc_tpad(T);
    p.K = K;
    p.N = N;
    p.G = K / kGroup;
    p.RT = N / kTileRows;
    p.RB = (N + kTcRows - 1) / kTcRows;
    int ks = num_sms / (p.RB > 0 ? p.RB : 1);
    const int sg = tc_stage_groups(p.TP);
    const int max_ks = p.G / (2 * sg) > 0 ? p.G / (2 * sg) : 1;  // >= 2 stages a piece
    if (ks > max_ks) ks = max_ks;
    if (ks < 1) ks = 1;
    p.KS = ks;
    p.P = p.RB * p.KS;
    p.stages = tc_stages(bits, p.TP);
    p.smem_bytes = p.stages * tc_stage_bytes(bits, p.TP) + tc_extra_bytes(p.TP);
    return p.stages >= 2 && p.G > 0;
}

struct TcArgs {                // aligned as CUtensorMap requires
    CUtensorMap xmap;        // X viewed as [K/64][T][64] bf16 (tokens past T read as zeros)
    CUtensorMap wmap;        // packed codes viewed as [RT][G][tile bytes / 8] (8-byte elements)
    CUtensorMap smap;        // packed scales viewed as [RT][G][4] (8-byte elements)
    const uint8_t* W;        // packed codes
    const uint8_t* S;        // packed scales
    uint16_t* Y;             // bf16 [T][N] (output modes kTcOutY and kTcOutSwiglu)
    float* G;                // fp32 [T][N]: written (kTcOutGate) or read (kTcOutSwiglu)
    float gscale;            // NVFP4 tensor scale (applied with each group partial), else 1
    float* partials;         // RB * KS slots of kTcRows x TP floats (K split only)
    int* tickets;            // one per row block, zero between calls
    int* dev_err;
    unsigned long long wait_ns;
    TcPlan p;
};

// ---------------------------------------------------------------- tcgen05 helpers

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// The A-fragment registers of a lane for the four K steps of a group (rows r, r+8; K pairs
// c, c+4 of each 16-wide step; 16 registers) into TMEM: step j's registers land at lanes
// taddr.lane + r, + r + 8 and columns taddr.col + 8 j + c, + 8 j + 4 + c, i.e. 64 K in natural
// order across 32 columns of 16 lanes (the 16x128b pattern repeated 8 times along columns).
__device__ __forceinline__ void tmem_st_group(uint32_t taddr, const uint32_t (&a)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(a[8]), "r"(a[9]),
        "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15])
        : "memory");
}
// Two consecutive groups (64 columns) with one store: the 16x128b pattern repeated 16 times,
// the first group's registers, then the second's.
__device__ __forceinline__ void tmem_st_pair(uint32_t taddr, const uint32_t (&a)[16], const uint32_t (&b)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x128b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(a[8]), "r"(a[9]),
        "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15]), "r"(b[0]), "r"(b[1]), "r"(b[2]),
        "r"(b[3]), "r"(b[4]), "r"(b[5]), "r"(b[6]), "r"(b[7]), "r"(b[8]), "r"(b[9]), "r"(b[10]), "r"(b[11]), "r"(b[12]),
        "r"(b[13]), "r"(b[14]), "r"(b[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 consecutive columns of the thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t v[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// D (+)= A * B: M = 128, N from idesc, K = 16; A in TMEM, B through a shared-memory descriptor.
// Issued by the lanes whose `issue` is true (one lane), with the whole warp executing the
// instruction so that no branch surrounds it.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate, bool issue) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"((uint32_t)issue)
        : "memory");
}

// Arrive once on an mbarrier when all tcgen05 operations the issuing lane issued so far are done
// (predicated like tc_mma).
__device__ __forceinline__ void tc_commit(uint32_t bar, bool issue) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
        "r"((uint32_t)issue)
        : "memory");
}

// Shared-memory descriptor of a K-major operand in the 128-byte swizzled layout: rows of 128
// bytes (64 bf16 of K), 8-row atoms of 1024 bytes (the stride between 8-row groups), atoms
// 1024-byte aligned. A K step of 16 starts 32 bytes further into the row.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor: D fp32, A and B bf16, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                 uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}


__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// K step J of a lane's code word as four bf16x2 registers holding (q - z) 2^-12 exactly: the
// offset code is placed under the bf16 exponent of 2^-5 (fraction unit 2^-12), so a register
// holds 2^-5 + q 2^-12, and subtracting 2^-5 + z 2^-12 leaves (q - z) 2^-12, representable.
template <int BITS, int J>
__device__ __forceinline__ void tc_decode(const uint4& w, uint32_t hb, uint32_t a[4]) {
    constexpr uint32_t kMagic = 0x3D003D00u;                          // 2^-5 in both halves
    constexpr uint32_t kOff = BITS == 4 ? 0x3D083D08u : 0x3D103D10u;  // 2^-5 + z 2^-12
    uint32_t magic;
    asm("mov.b32 %0, %1;" : "=r"(magic) : "n"(kMagic));
    const uint32_t word = J == 0 ? w.x : (J == 1 ? w.y : (J == 2 ? w.z : w.w));
    if constexpr (BITS == 4)
        decode_q4_bf16(word, a, magic);
    else
        decode_q5_bf16<J>(word, hb, a, magic);
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = bf16x2_sub(a[i], kOff);
}

// K step of a lane's NVFP4 code word (w: registers 0..3 of the mma.sync A fragment, rows r,
// r + 8; sc: the e4m3 block scales of rows r (low byte) and r + 8) as four bf16x2 registers
// holding e2m1 x e4m3 x 2^-20, exactly: the fp16 product has at most 6 significant bits and is
// exact in bf16, and |e2m1 x e4m3| <= 2688 keeps 64 products with any finite bf16 activation
// below 2^126 once scaled by 2^-20.
__device__ __forceinline__ void tc_decode_fp4(uint32_t w, uint32_t sc, uint32_t a[4]) {
    decode_fp4(w, sc, a);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = *reinterpret_cast<const __half2*>(&a[i]);
        const float2 f = __half22float2(h);
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * 0x1p-20f, f.y * 0x1p-20f);
        a[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
}

// One lane of a full warp returns true (the same lane every time the whole warp calls it).
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\telect.sync rx|px, %1;\n\tselp.b32 %0, 1, 0, px;\n\t}"
                 : "=r"(pred)
                 : "r"(0xFFFFFFFFu));
    return pred != 0;
}

// ---------------------------------------------------------------- the kernel

template <int BITS, int TP, int MODE>
__global__ void __launch_bounds__(tc_threads(BITS, TP), 1) tc_proj_kernel(const __grid_constant__ TcArgs a) {
    extern __shared__ __align__(1024) uint8_t tc_smem[];
    uint8_t* const smem = tc_smem;
    constexpr int TB = BITS == 5 ? kQ5TileBytes : kQ4TileBytes;
    constexpr int BG = tc_stage_groups(TP);
    static_assert(BG % kTcPair == 0, "decoder pairs tile a stage");
    constexpr int STB = scale_tile_bytes(BITS);
    constexpr bool FP4 = BITS == kFp4;
    constexpr int kWBytes = kTcTiles * BG * (TB + STB);     // codes, then scales
    constexpr int kWRegion = tc_weight_region(BITS, TP);    // padded: X starts 1024-aligned
    constexpr int kXBytes = TP * BG * kGroup * 2;
    constexpr int kStageBytes = kWRegion + kXBytes;
    static_assert(kWRegion % 1024 == 0 && kWRegion >= kWBytes && (TP * 128) % 1024 == 0,
                  "activation blocks on 1024-byte boundaries");
    constexpr uint32_t kCols = kTcCols;
    // TMEM columns of an A buffer (a stage) and of a P buffer (kPG groups: one MMA-to-epilogue
    // hand-off; three groups where two such buffers still fit, TP = 16: fewer hand-offs, 18.1
    // -> 17.7 us at T = 16 on the decode shape); two P buffers at every TP
    constexpr int kPG = (TP == 16 && BG % 3 == 0) ? 3 : kTcPair, kPSteps = BG / kPG;
    static_assert(BG % kPG == 0, "P steps tile a stage");
    constexpr int kAStage = BG * 32, kPCols = kPG * TP;
    constexpr int kP = (kTcCols - kTcA * kAStage) / kPCols;
    static_assert(kP >= 2 && kP <= kTcMaxP, "TMEM budget");
    constexpr uint32_t kIdesc = tc_idesc_bf16(TP);
    constexpr int kDec = tc_decoders(BITS, TP), kEpi = tc_epilogues(BITS, TP);
    constexpr int kDecPerTile = kDec / kTcTiles;     // warps sharing a tile's groups
    constexpr int kMmaWarp = 1 + kDec, kEpi0 = kMmaWarp + kTcIssuers;  // first issuer, first epilogue warp

    const TcPlan& p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int nstages = tc_stages(BITS, TP);      // compile time: no division in the loops
    const int rb = (int)blockIdx.x / p.KS, kp = (int)blockIdx.x % p.KS;
    const int g0 = (int)((long long)kp * p.G / p.KS), g1 = (int)((long long)(kp + 1) * p.G / p.KS);
    const int ngroups = g1 - g0;
    const int nst = (ngroups + BG - 1) / BG;          // stages this block streams
    const int nsteps = (ngroups + kPG - 1) / kPG;    // P steps
    const uint64_t wait_ns = a.wait_ns;

    uint8_t* stage_mem = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage_mem + nstages * kStageBytes);
    // bars: full[S], empty[S], a_full[A], a_empty[A], p_full[P], p_empty[P], done; then flags
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * kTcMaxStages;
    const uint32_t afull0 = empty0 + 8 * kTcMaxStages, aempty0 = afull0 + 8 * kTcA;
    const uint32_t pfull0 = aempty0 + 8 * kTcA, pempty0 = pfull0 + 8 * kTcMaxP, done_bar = pempty0 + 8 * kTcMaxP;
    volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * kTcMaxStages + 2 * kTcA + 2 * kTcMaxP + 1);
    // flags: [0] abort, [1] stages issued, [2] producer done, [3] TMEM base, [4] last ticket

    if (tid == 0) {
        for (int i = 0; i < nstages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kDec + kTcIssuers + kEpi);
        }
        for (int i = 0; i < kTcA; ++i) {
            mbar_init(afull0 + 8 * i, kDec);
            mbar_init(aempty0 + 8 * i, kTcIssuers);
        }
        for (int i = 0; i < kP; ++i) {
            mbar_init(pfull0 + 8 * i, 1);
            mbar_init(pempty0 + 8 * i, kEpi);
        }
        mbar_init(done_bar, kTcIssuers);
        flags[0] = 0;
        flags[1] = 0;
        flags[2] = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(const_cast<int*>(flags) + 3), kCols);
    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)flags[3];
    const uint32_t a_col0 = 0, p_col0 = kTcA * kAStage;

    // P step k covers groups kPG k .. kPG k + kPG - 1 of the block (the last may be past its
    // end), all in stage k / kPSteps from position gs0 = kPG (k % kPSteps).
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int it = 0;
            bool ok = true;
            for (int si = 0; si < nst && ok; ++si) {
                const int st = si % nstages;
                if (si >= nstages && !mbar_wait(empty0 + 8 * st, ((si / nstages) - 1) & 1, flags, a.dev_err, wait_ns)) {
                    ok = false;
                    break;
                }
                const int g = g0 + si * BG;
                uint8_t* sb = stage_mem + st * kStageBytes;
                const uint32_t fb = full0 + 8 * st;
                mbar_arrive_expect_tx(fb, (uint32_t)(kWBytes + kXBytes));  // whole boxes, zeros included
                tma_load_3d_hint(smem_u32(sb), &a.wmap, 0, g, rb * kTcTiles, fb, pol);
                tma_load_3d_hint(smem_u32(sb + kTcTiles * BG * TB), &a.smap, 0, g, rb * kTcTiles, fb, pol);
                // the weights are never written by a kernel that lets its dependents start
                // early; X may be the preceding kernel's output
                if (si == 0) grid_dependency_wait();
                tma_load_3d(smem_u32(sb + kWRegion), &a.xmap, 0, 0, g, fb);
                ++it;
            }
            if (!ok) {
                const int first = it > nstages ? it - nstages : 0;
                for (int j = first; j < it; ++j)
                    mbar_wait_drain(full0 + 8 * (j % nstages), (j / nstages) & 1, kDrainNs);
            }
            flags[1] = it;
            __threadfence_block();
            flags[2] = 1;
        }
    } else if (warp <= kDec) {
        // ------------------------------------------------------------ decoders
        const int q = warp & 3;                        // TMEM lane quarter
        const int h = ((warp - 1) >> 2) & 1;           // which half of it
        const int e = (warp - 1) >> 3;                 // which of the tile's decoders
        const int m = 2 * q + h;                       // the warp's 16-row tile of the block
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q + 16 * h) << 16) + a_col0;
        // Group gs of stage st (position gs of the stage) into the lane's 16 A-fragment registers.
        auto decode_group = [&](int st, int gs, uint32_t (&r)[16]) {
            const uint8_t* code = stage_mem + st * kStageBytes + m * BG * TB + gs * TB + lane * 16;
            const uint4 w = *reinterpret_cast<const uint4*>(code);
            if constexpr (FP4) {
                // the lane's 8 block-scale bytes: rows r, r + 8 for each K step
                const uint2 sc = *reinterpret_cast<const uint2*>(stage_mem + st * kStageBytes + kTcTiles * BG * TB +
                                                                 m * BG * STB + gs * STB + (lane >> 2) * 8);
                tc_decode_fp4(w.x, sc.x, r + 0);
                tc_decode_fp4(w.y, sc.x >> 16, r + 4);
                tc_decode_fp4(w.z, sc.y, r + 8);
                tc_decode_fp4(w.w, sc.y >> 16, r + 12);
            } else {
                const uint32_t hb = BITS == 5 ? *reinterpret_cast<const uint32_t*>(code + 512 - lane * 12) : 0u;
                tc_decode<BITS, 0>(w, hb, r + 0);
                tc_decode<BITS, 1>(w, hb, r + 4);
                tc_decode<BITS, 2>(w, hb, r + 8);
                tc_decode<BITS, 3>(w, hb, r + 12);
            }
        };
        // Groups gl, gl + 1 of the block (those inside its range), at positions gl % BG of stage st.
        auto decode_pair = [&](int st, int gl, uint32_t (&r)[kTcPair][16]) {
#pragma unroll
            for (int gp = 0; gp < kTcPair; ++gp) {
                if (gl + gp >= ngroups) break;
                decode_group(st, (gl + gp) % BG, r[gp]);
            }
        };
        // One register set per group of the stage that the warp decodes: none is rewritten while
        // its store may be in flight. One decoder per tile: pairs of groups (both decoded, then
        // both stored); two: every other group, each stored once decoded.
        constexpr int kMine = BG / kDecPerTile;
        static_assert(BG % kDecPerTile == 0 && (kDecPerTile == 1 || kDecPerTile == 2), "decoders split a stage");
        uint32_t r[kDecPerTile == 1 ? BG / kTcPair : 1][kTcPair][16];   // one decoder per tile
        uint32_t r1[kDecPerTile == 1 ? 1 : kMine][16];                   // two decoders per tile
        bool ok = true;
        for (int si = 0; si < nst; ++si) {
            // one stage per hand-off: its BG groups go to A buffer si % kTcA (32 columns a group)
            const int st = si % nstages, ab = si % kTcA, gl = si * BG;
            ok = mbar_wait(full0 + 8 * st, (si / nstages) & 1, flags, a.dev_err, wait_ns) && ok;
            if (si >= kTcA) ok = mbar_wait(aempty0 + 8 * ab, ((si / kTcA) - 1) & 1, flags, a.dev_err, wait_ns) && ok;
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (ok) {
                const uint32_t base = lane_base + kAStage * ab;
                if constexpr (kDecPerTile == 1) {
#pragma unroll
                    for (int pr = 0; pr < BG / kTcPair; ++pr) {
                        // a pair decodes while the stores of the pairs before it complete
                        const int g = gl + kTcPair * pr;
                        decode_pair(st, g, r[pr]);
                        // one store per pair for 4-bit codes and NVFP4 at TP = 16 and 64 (decode
                        // shape: T = 16 17.7 -> 16.5 us, T = 64 21.7 -> 20.7, NVFP4 T = 64 29.8 ->
                        // 29.3); at TP = 32 (18.6 -> 18.7) and for 5-bit codes (+1-2 %) slower
                        static_assert(kTcPair == 2, "one store per pair of groups");
                        if (BITS != 5 && TP != 32 && g + 1 < ngroups) {
                            tmem_st_pair(base + 32 * (kTcPair * pr), r[pr][0], r[pr][1]);
                        } else {
#pragma unroll
                            for (int gp = 0; gp < kTcPair; ++gp)
                                if (g + gp < ngroups) tmem_st_group(base + 32 * (kTcPair * pr + gp), r[pr][gp]);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kMine; ++j) {
                        // a group decodes while the stores of the groups before it complete
                        const int gs = kDecPerTile * j + e;
                        if (gl + gs < ngroups) {
                            decode_group(st, gs, r1[j]);
                            tmem_st_group(base + 32 * gs, r1[j]);
                        }
                    }
                }
            }
            __syncwarp();
            mbar_arrive_if(empty0 + 8 * st, lane == 0);  // the stage's codes are all in registers
            if (ok) tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            mbar_arrive_if(afull0 + 8 * ab, lane == 0);
        }
    } else if (warp < kEpi0) {
        // ------------------------------------------------------------ MMA issuers
        // Issuer i takes the P steps k with k % kTcIssuers == i. Every issuer waits for every
        // stage and, after its P steps of the stage, commits the stage's A buffer and shared
        // memory (those barriers count one arrival per issuer).
        const int iss = warp - kMmaWarp;
        bool ok = true;
        for (int si = 0; si < nst && ok; ++si) {
            const int st = si % nstages, ab = si % kTcA;
            ok = mbar_wait(full0 + 8 * st, (si / nstages) & 1, flags, a.dev_err, wait_ns);
            ok = ok && mbar_wait(afull0 + 8 * ab, (si / kTcA) & 1, flags, a.dev_err, wait_ns);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t xbase = smem_u32(stage_mem + st * kStageBytes + kWRegion);
            const uint32_t a0 = tmem + a_col0 + kAStage * ab;
            const bool leader = elect_one();
#pragma unroll
            for (int hh = 0; hh < kPSteps; ++hh) {
                const int k = kPSteps * si + hh;         // P step: groups kPG k .. kPG k + kPG - 1
                if (k >= nsteps) break;
                if (k % kTcIssuers != iss) continue;
                const int pb = k % kP;
                if (k >= kP) ok = mbar_wait(pempty0 + 8 * pb, ((k / kP) - 1) & 1, flags, a.dev_err, wait_ns);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d0 = tmem + p_col0 + kPCols * pb;
#pragma unroll
                for (int gp = 0; gp < kPG; ++gp) {
                    if (kPG * k + gp >= ngroups) break;
                    const int gs = kPG * hh + gp;        // position in the stage
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // K step j of group gs: bytes 32 j .. 32 j + 31 of the group block's rows
                        const uint64_t bd = smem_desc_sw128(xbase + (uint32_t)(gs * TP * 128 + 32 * j));
                        tc_mma(d0 + TP * gp, a0 + 32 * gs + 8 * j, bd, kIdesc, j > 0 ? 1u : 0u, leader);
                    }
                }
                tc_commit(pfull0 + 8 * pb, leader);
            }
            if (!ok) break;
            tc_commit(aempty0 + 8 * ab, leader);
            tc_commit(empty0 + 8 * st, leader);
        }
        // every MMA of both issuers has completed before TMEM can be freed
        const bool leader = elect_one();
        tc_commit(done_bar, leader);
        mbar_wait_drain(done_bar, 0, kDrainNs);
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = 32 * q + lane;                 // row of the block = TMEM lane
        const int m = row >> 4, rr = row & 15;
        const int sidx = 2 * (rr & 7) + (rr >> 3);     // the row's place in a packed scale tile
        constexpr int kTok = TP / (kEpi / 4);          // tokens of one epilogue warp: t0 .. t0 + kTok - 1
        const int t0 = kEpi == 4 ? 0 : kTok * ((warp - kEpi0) >> 2);
        grid_dependency_wait();                        // Y, G, partials and tickets may be in use before
        float acc[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i) acc[i] = 0.f;
        constexpr int kChunk = kTok < 32 ? kTok : 32;  // columns loaded before one wait
        for (int k = 0; k < nsteps; ++k) {
            const int si = k / kPSteps, hh = k % kPSteps, gs0 = kPG * hh, st = si % nstages;
            const int pb = k % kP;
            const bool last = hh == kPSteps - 1 || k == nsteps - 1;
            bool ok = true;
            if (hh == 0) ok = mbar_wait(full0 + 8 * st, (si / nstages) & 1, flags, a.dev_err, wait_ns);
            ok = mbar_wait(pfull0 + 8 * pb, (k / kP) & 1, flags, a.dev_err, wait_ns) && ok;
            tc_fence_after();
            if (ok) {
                const uint8_t* sc = stage_mem + st * kStageBytes + kTcTiles * BG * TB + m * BG * STB;
                const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + p_col0 + kPCols * pb + t0;
#pragma unroll
                for (int gp = 0; gp < kPG; ++gp) {
                    if (kPG * k + gp >= ngroups) break;
                    // NVFP4: the block scales are in the decoded weights, which carry 2^-20; the
                    // tensor scale g joins 2^20 here (exact), so that a partial is never
                    // scaled up past what g brings back down
                    const float s = FP4 ? (float)(1 << kTcFp4ScaleExp) * a.gscale
                                        : __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(
                                              sc + (gs0 + gp) * kScaleTileBytes + 2 * sidx))) *
                                              (float)(1 << kTcScaleExp);
#pragma unroll
                    for (int c = 0; c < kTok; c += kChunk) {
                        uint32_t v[kChunk];
#pragma unroll
                        for (int c2 = 0; c2 < kChunk; c2 += 16) tmem_ld16(base + TP * gp + c + c2, v + c2);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < kChunk; ++i) acc[c + i] = fmaf(s, __uint_as_float(v[i]), acc[c + i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            mbar_arrive_if(pempty0 + 8 * pb, lane == 0);
            mbar_arrive_if(empty0 + 8 * st, lane == 0 && last);
        }
        // outputs: rows past N and tokens past T are not stored. The four epilogue warps agree on
        // whether the block aborted before any of them enters the barriers below.
        const int nrow = rb * kTcRows + row;
        auto store = [&](int t, float v) {
            const size_t i = (size_t)t * p.N + nrow;
            if constexpr (MODE == kTcOutGate)
                a.G[i] = v;
            else if constexpr (MODE == kTcOutSwiglu)
                a.Y[i] = bf16_bits_rn(silu_mul(__ldcg(a.G + i), v));
            else
                a.Y[i] = bf16_bits_rn(v);
        };
        if (!named_bar_or(1, kEpi * 32, flags[0] != 0)) {
            if (p.KS == 1) {
                if (nrow < p.N) {
#pragma unroll
                    for (int i = 0; i < kTok; ++i)
                        if (t0 + i < p.T) store(t0 + i, acc[i]);
                }
            } else {
                float* part = a.partials + ((size_t)rb * p.KS + kp) * (kTcRows * TP);
#pragma unroll
                for (int i = 0; i < kTok; ++i) part[(t0 + i) * kTcRows + row] = acc[i];
                named_bar_sync(1, kEpi * 32);          // the block's partial is complete
                const int leader = kEpi0 * 32;
                if (tid == leader) {
                    fence_acq_rel_gpu();
                    flags[4] = ticket_add(a.tickets + rb) == p.KS - 1;
                }
                named_bar_sync(1, kEpi * 32);
                if (flags[4]) {
                    fence_acq_rel_gpu();
                    float sum[kTok];
#pragma unroll
                    for (int i = 0; i < kTok; ++i) sum[i] = 0.f;
                    for (int k2 = 0; k2 < p.KS; ++k2) {   // fixed order: deterministic
                        const float* src = a.partials + ((size_t)rb * p.KS + k2) * (kTcRows * TP);
#pragma unroll
                        for (int i = 0; i < kTok; ++i) sum[i] += __ldcg(src + (t0 + i) * kTcRows + row);
                    }
                    if (nrow < p.N) {
#pragma unroll
                        for (int i = 0; i < kTok; ++i)
                            if (t0 + i < p.T) store(t0 + i, sum[i]);
                    }
                    if (tid == leader) a.tickets[rb] = 0;
                }
            }
        }
    }

    if (flags[0] && tid == 0) {
        // Aborted: wait (bounded) for the producer to stop, then for its last copy into each stage.
        const uint64_t t0 = global_timer_ns();
        while (!flags[2] && global_timer_ns() - t0 < 2 * kDrainNs) {
        }
        const int issued = flags[1];
        for (int j = issued > nstages ? issued - nstages : 0; j < issued; ++j)
            mbar_wait_drain(full0 + 8 * (j % nstages), (j / nstages) & 1, kDrainNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

// ---------------------------------------------------------------- host launch

// One launch of tc_proj_kernel<BITS, TP, MODE>: a block per plan block, programmatic dependent launch
// when `pdl`. The shared-memory opt-in is set once per device and thread.
template <int BITS, int TP, int MODE = kTcOutY>
inline cudaError_t tc_launch(const TcArgs& a, cudaStream_t stream, bool pdl) {
    auto kern = tc_proj_kernel<BITS, TP, MODE>;
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
    cfg.blockDim = dim3(tc_threads(BITS, TP));
    cfg.dynamicSmemBytes = a.p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}


}  // namespace nq
