// nq_common.cuh -- layout constants, the work plan and PTX helpers shared by the kernels
// of the groupwise int4/int5 small-batch projection (sm_103a).
//
// Packed layout (this library's definition; the pages give none). A packed weight is two
// buffers, the codes Wq and the scales S, both cut into tiles of 16 output rows x one
// 64-wide K group, tile (rt, g) with rt = n / 16 and g = k / 64, stored row-tile-major
// (tile (rt, g) is number rt * G + g, G = K / 64):
//   Wq: TB bytes per tile (512 for Q4, 640 for Q5) at (rt * G + g) * TB. Inside a code
//       tile, lane l (0..31) of a warp owns 16 bytes = four uint32 words, one per 16-wide
//       K step j: the word holds the lane's A-operand fragment of an m16n8k16 tensor-core
//       MMA for that step, one LOP3 away per register (see decode_q4). Q5 code tiles append
//       one uint32 of high bits per lane (128 bytes per tile).
//   S:  32 bytes per tile (16 fp16 scales) at (rt * G + g) * 32, ordered (row r, row r+8)
//       for r = 0..7, so lane l reads one uint32 holding the scales of its rows l/4, l/4+8.
// A row tile's codes and scales are each contiguous along K, so a pipeline stage of any
// run of groups is one bulk copy of codes and one of scales per tile.
//
// NVFP4 weights (format tag kFp4) use the same tiles: a code tile holds 16 rows x 64 e2m1
// codes (512 B), lane l's word j holding its four A registers of K step j in bytes 0..3
// (register m's two codes in byte m, the even-K element in the low nibble); a scale tile
// holds the 16 x 4 e4m3 block scales (one per 16-wide K step, 64 B), byte 8 r + 2 j + h for
// row r + 8 h, so lane l reads its rows' scales of all four K steps as 8 bytes at 8 (l/4).
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define NQ_HD __host__ __device__ __forceinline__
#else
#define NQ_HD inline
#endif

namespace nq {

constexpr int kGroup = 64;           // K elements per scale group
constexpr int kTileRows = 16;        // output rows per tile (MMA M)
constexpr int kQ4TileBytes = 512;    // 16 x 64 nibbles
constexpr int kQ5TileBytes = 640;    // + 16 x 64 high bits
constexpr int kScaleTileBytes = 32;  // 16 fp16
constexpr int kFp4 = 14;             // format tag of NVFP4 weights (template argument BITS)
constexpr int kFp4ScaleTileBytes = 64;  // 16 rows x 4 e4m3 block scales
#ifndef NQ_BLOCK_GROUPS
#define NQ_BLOCK_GROUPS 32
#endif
constexpr int kBlockGroups = NQ_BLOCK_GROUPS;  // groups per pipeline stage (stages start on multiples of it)
#ifndef NQ_CONSUMER_WARPS
#define NQ_CONSUMER_WARPS 8
#endif
constexpr int kConsumerWarps = NQ_CONSUMER_WARPS;
constexpr int kProducerWarp = kConsumerWarps;         // issues the bulk copies
constexpr int kEpilogueWarp = kConsumerWarps + 1;     // first of the warps that reduce runs,
constexpr int kEpilogueWarps = 2;                     // store them and settle split-K (runs alternate)
constexpr int kThreads = (kConsumerWarps + 1 + kEpilogueWarps) * 32;
constexpr int kChunkGroups = kBlockGroups;           // K groups per pipeline stage
constexpr int kGroupsPerWarp = kChunkGroups / kConsumerWarps;
static_assert(kGroupsPerWarp * kConsumerWarps == kChunkGroups, "stage groups split evenly over warps");
constexpr int kMaxStages = 12;
constexpr int kSmemLimit = 227 * 1024;
// Weight bytes that must be in flight to keep HBM busy (bandwidth x loaded latency, about
// 6.8 TB/s x 1.2 us), measured: whole-pair grids below it streamed slower than stream-K.
constexpr long long kSaturateBytes = 8ll << 20;
constexpr int kXBudget = 97 * 1024;  // on-chip activation slab (96 groups x 8 rows + padding)
constexpr int kMinUnitsPerCta = 16;
constexpr int kPartialFloats = 256;  // 2 M tiles x 16 rows x 8 tokens
constexpr int kMaxRed = 4;           // most run hand-over buffers (consumers -> epilogue warps)
constexpr int kRedBufBytes = kConsumerWarps * 2 * 512;  // one buffer: every warp's two accumulator tiles
constexpr long long kWaitTimeoutNs = 2000000000LL;  // default bound of a device-side wait: 2 s
constexpr unsigned long long kDrainNs = 100000000ull;  // bound of each wait for copies in flight on abort
// Bounds below this poll the barrier without suspending (mbarrier.test_wait), so that they
// are exact; longer bounds use the suspending mbarrier.try_wait, whose own hardware time
// limit is far below this.
constexpr unsigned long long kPollBelowNs = 1000000ull;
constexpr int kMaxCluster = 4;       // most K slabs handled by one thread-block cluster
constexpr int kSliceT = 8;           // tokens one projection launch handles (MMA N = 8)
constexpr int kMaxT = 64;            // tokens one projection call accepts (kSliceT per launch)

// Errors a kernel can raise through the workspace flag word.
constexpr int kDevErrTimeout = 1;

NQ_HD int tpad(int T) { return T <= 1 ? 1 : (T <= 2 ? 2 : (T <= 4 ? 4 : 8)); }

// Byte offsets inside a packed weight (TB = code bytes per tile, 512 or 640).
NQ_HD long long packed_code_off(int rt, int g, int G, int TB) { return ((long long)rt * G + g) * TB; }
NQ_HD constexpr int code_tile_bytes(int bits) { return bits == 5 ? kQ5TileBytes : kQ4TileBytes; }
NQ_HD constexpr int scale_tile_bytes(int bits) { return bits == kFp4 ? kFp4ScaleTileBytes : kScaleTileBytes; }
NQ_HD long long packed_scale_off(int rt, int g, int G, int STB) { return ((long long)rt * G + g) * STB; }

// The work split of one projection call. One "unit" is one 64-wide K group of one row pair
// (two 16-row tiles; for SwiGLU the gate tile and the up tile of the same rows). Units are
// ordered slab-major: for each K slab, for each pair, the slab's groups. The persistent
// grid of P blocks takes equal contiguous ranges of units ("stream-K"), so every block
// streams the same number of weight bytes whatever the shape.
struct Plan {
    int bits, mode, T, TP, K, N, G, RT, RP;
    int GS, S;             // groups per slab (last slab may be shorter), slab count
    long long U;           // units (< 2^31 for every accepted shape)
    int P;                 // blocks
    int Uq, Ur;            // U = Uq * P + Ur: block c owns Uq units, plus one if c < Ur
    int CG, stages;
    long long slots;       // partial-sum slots: S * RP + P
    int tile_bytes, stage_bytes, x_bytes, corr_bytes, red_bytes, bar_bytes, smem_bytes;
    int f16;               // 1: fp16 MMA operands (X converted in shared memory), 0: bf16
    int nred;              // run hand-over buffers (2..kMaxRed)
    int cl;                // 1, or S: slab clusters (block rank r of a cluster takes slab r)
    int cl_bytes;          // cluster exchange buffers at the end of shared memory (0 if cl == 1)
};

// Shared-memory bytes of the exchange buffers of a slab cluster of S blocks: per epilogue
// warp, one partial run of each non-leading rank.
NQ_HD int cluster_buffer_bytes(int S) { return S > 1 ? kEpilogueWarps * (S - 1) * kPartialFloats * 4 : 0; }

// Largest T that uses fp16 operands: one shift per code word instead of three, paid for by
// converting the activation slab to fp16 once per block, which grows with T.
#ifndef NQ_F16_MAX_T
#define NQ_F16_MAX_T 2
#endif

// Shared-memory layout of a plan whose slab geometry (GS) is set: activation slab,
// zero-point sums, run hand-over buffers, barriers, cluster buffers (p.cl_bytes) and as many
// pipeline stages as fit. Returns the stage count.
NQ_HD int plan_smem(Plan& p) {
    const int Tr = p.T > 0 ? p.T : 1;
    p.CG = kChunkGroups;
    p.tile_bytes = code_tile_bytes(p.bits);
    p.stage_bytes = 2 * p.CG * (p.tile_bytes + scale_tile_bytes(p.bits));
    p.x_bytes = (Tr * (p.GS * 128 + 16) + 16 + 127) / 128 * 128;  // T rows of pitch GS*128+16, zero row
    p.corr_bytes = (p.GS * 8 * 4 + 127) / 128 * 128;  // O[gl][8 tokens] fp32
    p.bar_bytes = 512;                           // barriers, flags, per-token range data
    // Run hand-over buffers: kMaxRed if they fit without costing a pipeline stage against
    // two, else two; spare buffers let the consumers run ahead of a split-K settle. The count
    // is a multiple of kEpilogueWarps, so each buffer is always served by the same epilogue
    // warp (two warps never wait on one buffer's barrier at once).
    static_assert(kMaxRed % kEpilogueWarps == 0 && 2 % kEpilogueWarps == 0, "buffers per epilogue warp");
    int st = 0;
    for (int nr = kMaxRed; nr >= 2; nr -= 2) {
        const int fixed = p.x_bytes + p.corr_bytes + nr * kRedBufBytes + p.bar_bytes + p.cl_bytes;
        int s2 = (kSmemLimit - fixed) / p.stage_bytes;
        if (s2 > kMaxStages) s2 = kMaxStages;
        const int fixed2 = p.x_bytes + p.corr_bytes + 2 * kRedBufBytes + p.bar_bytes + p.cl_bytes;
        int s_two = (kSmemLimit - fixed2) / p.stage_bytes;
        if (s_two > kMaxStages) s_two = kMaxStages;
        if (s2 == s_two || nr == 2) {
            p.nred = nr;
            st = s2;
            break;
        }
    }
    p.red_bytes = p.nred * kRedBufBytes;
    p.stages = st;
    p.smem_bytes = p.x_bytes + p.corr_bytes + p.red_bytes + p.bar_bytes + p.cl_bytes + st * p.stage_bytes;
    p.f16 = p.bits == kFp4 || p.T <= NQ_F16_MAX_T ? 1 : 0;  // NVFP4: fp16 weights at every T
    return st;
}

NQ_HD bool make_plan(int bits, int mode, int T, int K, int N, int num_sms, Plan& p) {
    p.bits = bits;
    p.mode = mode;
    p.T = T;
    p.TP = tpad(T);
    p.K = K;
    p.N = N;
    p.G = K / kGroup;
    p.RT = N / kTileRows;
    p.RP = mode ? p.RT : (p.RT + 1) / 2;
    // Largest slab whose T padded activation rows plus one zero row fit the X budget.
    const int Tr = T > 0 ? T : 1;
    int gs_max = ((kXBudget - 16) / Tr - 16) / 128 / kBlockGroups * kBlockGroups;
    if (gs_max < kBlockGroups) gs_max = kBlockGroups;
    p.S = (p.G + gs_max - 1) / gs_max;
    if (p.S < 1) p.S = 1;
    p.GS = (p.G + p.S - 1) / p.S;
    if (p.S > 1) p.GS = (p.GS + kBlockGroups - 1) / kBlockGroups * kBlockGroups;  // slabs on block edges
    p.U = (long long)p.RP * p.G;
    p.cl = 1;
    p.cl_bytes = 0;
    const int st = plan_smem(p);
    // Grid. Stream-K over all SMs by default. One slab and row pairs that divide evenly
    // into k <= 4 per block (k = the fewest that fit the SMs): give each block whole pairs,
    // so no pair is split and no split-K settle (several L2 round trips at the end of a
    // short kernel) is needed, provided those blocks' rings can still keep HBM busy, i.e.
    // hold kSaturateBytes in flight, or the whole problem. With more pairs per block the
    // stream-K settles come early and overlap the stream, and the SMs a whole-pair grid
    // leaves idle cost more (measured: 8 pairs per block on 136 SMs, +3 to +4 %).
    long long P = p.U / kMinUnitsPerCta;
    if (P > num_sms) P = num_sms;
    if (P < 1) P = 1;
    if (p.S == 1 && num_sms > 0 && st > 0) {
        const int k = (p.RP + num_sms - 1) / num_sms;
        if (k >= 1 && k <= 4 && p.RP % k == 0) {
            const long long in_flight = (long long)(p.RP / k) * st * p.stage_bytes;
            const long long weights = p.U * 2 * (p.tile_bytes + scale_tile_bytes(p.bits));
            if (in_flight >= kSaturateBytes || in_flight >= weights) P = p.RP / k;
        }
    }
    p.P = (int)P;
    p.Uq = (int)(p.U / p.P);
    p.Ur = (int)(p.U % p.P);
    p.slots = (long long)p.S * p.RP + p.P;
    return st >= 2;
}

// Slab clusters (K split into S = 2..kMaxCluster slabs, bf16 operands): a thread-block
// cluster of S blocks per range of work, block rank r taking slab r of every row pair in
// the range, so each block stages one activation slab once and the S partial sums of a run
// are added on chip (rank 0 gathers them through distributed shared memory) instead of
// through the split-K workspace. p: the real plan (slab geometry, shared memory, P = C x S
// blocks). q: the cluster-level plan, one virtual slab of GS groups with stream-K over the C
// clusters; its segments, ticket counts and partial slots are those of the clusters, and a
// virtual segment maps to rank r's real groups by rank_segment.
NQ_HD bool make_cluster_plans(int bits, int mode, int T, int K, int N, int clusters, Plan& p, Plan& q) {
    if (!make_plan(bits, mode, T, K, N, 1, p)) return false;
    const int S = p.S;
    if (S < 2 || S > kMaxCluster || clusters < 1 || p.f16) return false;
    // Equal slabs on multiples of the consumer warp count (warp w consumes the groups that
    // are w modulo kConsumerWarps from the slab start); never larger than the plain slabs.
    int gs = (p.G + S - 1) / S;
    gs = (gs + kConsumerWarps - 1) / kConsumerWarps * kConsumerWarps;
    if ((long long)(S - 1) * gs >= p.G || gs > p.GS) return false;
    p.GS = gs;
    p.cl = S;
    p.cl_bytes = cluster_buffer_bytes(S);
    if (plan_smem(p) < 2) return false;
    q = p;
    q.K = gs * kGroup;
    q.G = gs;
    q.S = 1;
    q.GS = gs;
    q.U = (long long)q.RP * gs;
    q.P = (long long)clusters < q.U ? clusters : (int)q.U;
    q.Uq = (int)(q.U / q.P);
    q.Ur = (int)(q.U % q.P);
    q.slots = (long long)q.RP + q.P;
    p.P = q.P * S;
    p.U = (long long)p.RP * p.G;
    p.Uq = q.Uq;
    p.Ur = q.Ur;
    p.slots = q.slots;
    return true;
}

NQ_HD int slab_groups(const Plan& p, int s) { return s < p.S - 1 ? p.GS : p.G - (p.S - 1) * p.GS; }
NQ_HD long long slab_base(const Plan& p, int s) { return (long long)s * p.RP * p.GS; }
// Balanced split: the first Ur blocks own Uq + 1 units, the others Uq (32-bit arithmetic).
NQ_HD long long cta_begin(const Plan& p, int c) {
    return (long long)((unsigned)c * (unsigned)p.Uq + (unsigned)(c < p.Ur ? c : p.Ur));
}
// Block that owns unit u.
NQ_HD int cta_of(const Plan& p, long long u) {
    const unsigned uu = (unsigned)u, big = (unsigned)p.Ur * (unsigned)(p.Uq + 1);
    return uu < big ? (int)(uu / (unsigned)(p.Uq + 1)) : p.Ur + (int)((uu - big) / (unsigned)p.Uq);
}

// One run of consecutive units of one block inside one (slab, pair).
struct Segment {
    int s, rp, ga, gb;     // slab, pair, groups [ga, gb) in K-group numbering
    long long u_next;      // first unit after the segment
};

NQ_HD Segment segment_at(const Plan& p, long long u, long long u_end) {
    Segment sg;
    unsigned s = (unsigned)u / ((unsigned)p.RP * (unsigned)p.GS);
    if (s > (unsigned)(p.S - 1)) s = p.S - 1;
    sg.s = (int)s;
    const int gs = slab_groups(p, sg.s);
    const unsigned off = (unsigned)(u - slab_base(p, sg.s));
    sg.rp = (int)(off / (unsigned)gs);
    const int gl = (int)(off % (unsigned)gs);
    const long long run_end = slab_base(p, sg.s) + (long long)(sg.rp + 1) * gs;
    const long long e = run_end < u_end ? run_end : u_end;
    sg.ga = sg.s * p.GS + gl;
    sg.gb = sg.ga + (int)(e - u);
    sg.u_next = e;
    return sg;
}

// The segment after sg in the same block (runs after the first start at a slab's first
// group). Returns false when the block's range [.., u_end) is exhausted. No divisions.
NQ_HD bool segment_next(const Plan& p, Segment& sg, long long u_end) {
    const long long u = sg.u_next;
    if (u >= u_end) return false;
    if (sg.rp + 1 < p.RP) {
        sg.rp += 1;
    } else {
        sg.s += 1;
        sg.rp = 0;
    }
    const int gs = slab_groups(p, sg.s);
    const long long left = u_end - u;
    const int len = left < gs ? (int)left : gs;
    sg.ga = sg.s * p.GS;
    sg.gb = sg.ga + len;
    sg.u_next = u + len;
    return true;
}

// Processing order of a block's segments. With one slab, the (possibly partial) first and
// last runs go first, so their split-K partials are settled early and the block ends on a
// complete run; with several slabs every run is partial and the natural order keeps the
// activation slab loaded once per slab.
struct SegOrder {
    Segment first, last;   // natural first and last segment of the block
    int count;             // number of segments
};

NQ_HD SegOrder seg_order(const Plan& p, long long u0, long long u1) {
    SegOrder o;
    o.first = segment_at(p, u0, u1);
    o.last = o.first;
    o.count = 1;
    Segment sg = o.first;
    while (segment_next(p, sg, u1)) {
        o.last = sg;
        ++o.count;
    }
    return o;
}

// The i-th segment in processing order (i < count); `nat` is the natural-order iterator
// state used to walk the middle runs (call with i increasing by one from 0).
NQ_HD Segment seg_pick(const Plan& p, const SegOrder& o, int i, Segment& nat, long long u1) {
    if (p.S > 1 || o.count <= 2) {
        if (i == 0) nat = o.first; else segment_next(p, nat, u1);
        return nat;
    }
    if (i == 0) return o.first;
    if (i == 1) return o.last;
    if (i == 2) nat = o.first;
    segment_next(p, nat, u1);  // middle runs: natural segments 1 .. count-2
    return nat;
}

// Rank r's part of a cluster-level segment v (virtual groups [v.ga, v.gb) of one slab's
// width): the same groups of slab r, clipped to that slab (the last slab may be shorter,
// so the part may be empty).
NQ_HD Segment rank_segment(const Plan& p, const Segment& v, int r) {
    Segment sg = v;
    const int gs = slab_groups(p, r);
    sg.s = r;
    sg.ga = r * p.GS + (v.ga < gs ? v.ga : gs);
    sg.gb = r * p.GS + (v.gb < gs ? v.gb : gs);
    return sg;
}

// A segment that covers its whole pair (one slab, all K groups) is the pair's only
// contribution: its block writes the output directly.
NQ_HD bool segment_complete(const Plan& p, const Segment& sg) {
    return p.S == 1 && sg.ga == 0 && sg.gb == p.G;
}

// Number of (block, slab) runs that contribute to pair rp: the split-K fan-in.
NQ_HD int contributions(const Plan& p, int rp) {
    int c = 0;
    for (int s = 0; s < p.S; ++s) {
        const int gs = slab_groups(p, s);
        const long long a = slab_base(p, s) + (long long)rp * gs;
        c += cta_of(p, a + gs - 1) - cta_of(p, a) + 1;
    }
    return c;
}

// Partial-sum slot of the segment (s, rp) of block c. Unique because segments advance
// monotonically in both the run index s*RP+rp and the block index.
NQ_HD long long slot_of(const Plan& p, int s, int rp, int c) { return (long long)s * p.RP + rp + c; }

}  // namespace nq

#if defined(__CUDACC__)
#include <cuda_bf16.h>

namespace nq {

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// bf16 bits of v, round to nearest even.
__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// The SwiGLU epilogue in fp32: silu(g) * u = g / (1 + e^-g) * u.
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// One arrive by the lanes whose pred is true, issued by the whole warp with the predicate inside
// the instruction: no branch, so the warp does not reconverge behind the arrive (a branch around
// an arrive costs ~160 cycles per hand-off on sm_103 when the warp reconverges after it).
__device__ __forceinline__ void mbar_arrive_if(uint32_t bar, bool pred) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar),
        "r"((uint32_t)pred)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-suspending test of a phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase. Returns false (and raises the block's abort flag and
// the device error word) if the phase does not complete within limit_ns, or at once if the
// block has already aborted. Never spins forever.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* dev_err, uint64_t limit_ns) {
    const bool poll = limit_ns < kPollBelowNs;
    if (!poll && mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (*abort_flag) return false;
        if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(dev_err, kDevErrTimeout);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used to drain copies in flight before exit).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > limit_ns) return false;
    return true;
}

// ---------------------------------------------------------------- cluster helpers

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// 16-byte store into the shared memory of another block of the cluster that completes
// 16 transaction bytes on that block's mbarrier `bar` once the data is there (no fence).
__device__ __forceinline__ void cluster_store_async_v4(uint32_t addr, float a, float b, float c, float d,
                                                       uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
        "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d)),
        "r"(bar)
        : "memory");
}

// Arrive on an mbarrier of another block of the cluster, releasing this thread's earlier
// writes (and those it has observed) at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a phase completed by other blocks of the cluster (acquire at cluster
// scope). Same error behaviour as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  int* dev_err, uint64_t limit_ns) {
    const bool poll = limit_ns < kPollBelowNs;
    const uint64_t t0 = global_timer_ns();
    while (!(poll ? mbar_test_wait_cluster(bar, parity) : mbar_try_wait_cluster(bar, parity))) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(dev_err, kDevErrTimeout);
            return false;
        }
    }
    return true;
}

// Every thread of every block of the cluster (not .aligned: callers may have diverged).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One-dimensional bulk async copy global -> shared (TMA engine), completing on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// The same copy with no L2 eviction hint (activations: every block reads them).
__device__ __forceinline__ void bulk_g2s_plain(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier with an OR-reduction of a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Ticket for the split-K fix-up: one thread adds 1 with acquire-release semantics at GPU
// scope. Preceded by a block barrier, it publishes every thread's partial stores (release
// is cumulative); the last taker's acquire, followed by a block barrier, makes every
// earlier taker's partials visible to the whole block.
__device__ __forceinline__ int ticket_add(int* p) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
    return old;
}

// 16-byte asynchronous copy global -> shared through L2 (LSU path); both addresses 16-byte
// aligned. cp_async_wait_all waits for all of the thread's outstanding copies.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Acquire-release fence at GPU scope: orders this thread's earlier memory operations (and
// those it has observed) before its later ones, as seen by any thread on the GPU.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B (zero accumulator), m16n8k16, fp16 or bf16 inputs, fp32 results.
template <bool F16>
__device__ __forceinline__ void mma_zero_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    if constexpr (F16)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float d[4], const uint32_t a[4], uint32_t b0,
                                              uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- code decode
//
// The MMAs run on fp16 operands. fp16 0x6400 is 1024.0 with a unit step in its 10 fraction
// bits, so OR-ing a code q into bits 0..3 (or 0..4) of a half gives exactly 1024 + q, and
// OR-ing it into bits 4..7 gives exactly 1024 + 16 q. A lane's code word is laid out so that
// the codes of the fragment's lower-K pairs (registers 0, 1) sit at bits 0..3 and the codes
// of its upper-K pairs (registers 2, 3) at bits 4..7 of each half, after at most one shift:
//   word bits  0-3  a0 (row r,   k)       16-19 a1 (row r,   k+1)
//              4-7  a4 (row r,   k+8)     20-23 a5 (row r,   k+9)
//              8-11 a2 (row r+8, k)       24-27 a3 (row r+8, k+1)
//             12-15 a6 (row r+8, k+8)     28-31 a7 (row r+8, k+9)
// with r = lane/4 and k = 2*(lane%4) of the K step. The upper-K registers carry 16x their
// weight; the kernels store X / 16 at the upper-K positions of every 16-wide K step, so every
// product is (1024 + q) * x or (1024 + 16 q) * (x / 16) = (1024/16 ... ) exactly as wanted: the
// sum over a K step is sum(q * x) + 1024 * sum(x_lo + x_hi / 16), and the second term is the
// same MMA chain on the constant code 0 -- removed exactly by subtracting that chain.
constexpr uint32_t kF16Magic = 0x64006400u;   // 1024.0 in both halves

// (a & MASK) | c in one LOP3 (c is kept in a register so it is not split in two ops).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}

// Four fp16x2 A-fragment registers from one packed Q4 word: registers 0, 1 hold 1024 + q of
// the lower-K pairs, registers 2, 3 hold 1024 + 16 q of the upper-K pairs. One shift, four LOP3.
__device__ __forceinline__ void decode_q4(uint32_t w, uint32_t a[4], uint32_t magic = kF16Magic) {
    const uint32_t w8 = w >> 8;
    a[0] = and_or<0x000F000Fu>(w, magic);
    a[2] = and_or<0x00F000F0u>(w, magic);
    a[1] = and_or<0x000F000Fu>(w8, magic);
    a[3] = and_or<0x00F000F0u>(w8, magic);
}

// The same packed word decoded for bf16 operands (bf16 0x4300 = 128.0 with a unit step in its
// 7 fraction bits): every register holds 128 + q, so each code must sit at bits 0..3 of its
// half -- three shifts, four LOP3 -- and X is used as is (no division by 16).
constexpr uint32_t kBf16Magic = 0x43004300u;
__device__ __forceinline__ void decode_q4_bf16(uint32_t w, uint32_t a[4], uint32_t magic = kBf16Magic) {
    a[0] = and_or<0x000F000Fu>(w, magic);
    a[2] = and_or<0x000F000Fu>(w >> 4, magic);
    a[1] = and_or<0x000F000Fu>(w >> 8, magic);
    a[3] = and_or<0x000F000Fu>(w >> 12, magic);
}

// Q5 for bf16 operands: the high bit of every code goes to bit 4 of its half (+16).
template <int J>
__device__ __forceinline__ void decode_q5_bf16(uint32_t w, uint32_t h, uint32_t a[4], uint32_t magic = kBf16Magic) {
    a[0] = and_or<0x000F000Fu>(w, and_or<0x00100010u>(h << (4 - J), magic));
    a[2] = and_or<0x000F000Fu>(w >> 4, and_or<0x00100010u>(h >> J, magic));
    a[1] = and_or<0x000F000Fu>(w >> 8, and_or<0x00100010u>(h >> (4 + J), magic));
    a[3] = and_or<0x000F000Fu>(w >> 12, and_or<0x00100010u>(h >> (8 + J), magic));
}

// ---------------------------------------------------------------- NVFP4 decode
//
// Each A register is exact in fp16: an e2m1 element (at most 2 significant bits, 0.5 .. 6)
// times its e4m3 block scale (at most 4 significant bits, 2^-9 .. 448) has at most 6
// significant bits and lies inside fp16's normal range, so one fp16 multiply is exact.

// Two e2m1 codes (low byte of x, the first in bits 0..3) -> fp16x2.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t x) {
    uint32_t d;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(d) : "r"(x));
    return d;
}

// Two e4m3 values (low 16 bits of x, the first in bits 0..7) -> fp16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x) {
    uint32_t d;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(d) : "r"(x));
    return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The low (H0) or high (H1) half of x in both halves.
template <int H>
__device__ __forceinline__ uint32_t half_bcast(uint32_t x) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(x), "n"(H == 0 ? 0x1010 : 0x3232));
    return d;
}

// K step of an NVFP4 tile: w holds registers 0..3 in bytes 0..3 (rows r, r+8, r, r+8; lower
// then upper K pairs), sc the e4m3 scales of rows r (low byte) and r+8 (high byte).
__device__ __forceinline__ void decode_fp4(uint32_t w, uint32_t sc, uint32_t a[4]) {
    const uint32_t s2 = e4m3x2_to_f16x2(sc);
    const uint32_t s_r = half_bcast<0>(s2), s_r8 = half_bcast<1>(s2);
    a[0] = hmul2(e2m1x2_to_f16x2(w), s_r);
    a[1] = hmul2(e2m1x2_to_f16x2(w >> 8), s_r8);
    a[2] = hmul2(e2m1x2_to_f16x2(w >> 16), s_r);
    a[3] = hmul2(e2m1x2_to_f16x2(w >> 24), s_r8);
}

// Q5: as decode_q4, plus bit 4 of each code from the lane's high word h, which lands on bit 4
// of a lower-K half (+16) or bit 8 of an upper-K half (+256 = 16 * 16). For K step J the high
// bits of registers 0 / 2 sit at bits {J, 16+J} / {4+J, 20+J} of h and those of registers
// 1 / 3 at bits {8+J, 24+J} / {12+J, 28+J}: one left shift by 4-J aligns the first pair of
// registers, one right shift by 4+J the second.
template <int J>
__device__ __forceinline__ void decode_q5(uint32_t w, uint32_t h, uint32_t a[4], uint32_t magic = kF16Magic) {
    const uint32_t w8 = w >> 8;
    const uint32_t ha = h << (4 - J), hb = h >> (4 + J);
    a[0] = and_or<0x000F000Fu>(w, and_or<0x00100010u>(ha, magic));
    a[2] = and_or<0x00F000F0u>(w, and_or<0x01000100u>(ha, magic));
    a[1] = and_or<0x000F000Fu>(w8, and_or<0x00100010u>(hb, magic));
    a[3] = and_or<0x00F000F0u>(w8, and_or<0x01000100u>(hb, magic));
}

}  // namespace nq
#endif
