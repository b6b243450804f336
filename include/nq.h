/*
 * nq.h -- C ABI of the GB300 (sm_103a) groupwise int4/int5 small-batch projection library.
 *
 * The operation (what the pages tune for single-GPU decode and speculative verify rounds):
 *
 *     Y[t,n] = sum_k X[t,k] * W[k,n],   W[k,n] = s[n, k/64] * (q[n,k] - z),
 *     z = 8 for 4-bit codes (Q4), z = 16 for 5-bit codes (Q5),  t < T <= 64.
 *
 * Sources: "NInfer-4090" release post (lcz.me), section "V3 做了什么" -- small-batch Q4/Q5
 * projections with T=8 routing, used by the GDN projections, the attention Q5 projections
 * and the SwiGLU path; same post, section "实测数据" -- per-op timings of a T=8 attention Q5
 * gate/value projection and a GDN QK Q4 projection; "ninfer-ext" README, section
 * "与原版 NInfer 的对比" -- the Q5 K-split MMA path for small-batch verify rounds.
 * The pages give neither an API nor a storage format: both are this library's definition.
 *
 * Canonical layouts (host or device arrays; all little-endian):
 *   X    bf16   [T][K]     row-major activations
 *   Y, H bf16   [T][N]     row-major outputs (round to nearest even from fp32)
 *   Wq   uint32 [N][K/8]   Q4 codes: nibble i (bits 4i..4i+3) of word j is q[n, 8j+i]
 *   Wn   uint32 [N][K/8]   Q5 low nibbles, same rule
 *   Wh   uint32 [N][K/32]  Q5 high bits: bit i of word j is bit 4 of q[n, 32j+i]
 *   S    fp16   [N][K/64]  one scale per (output row n, 64-wide group of K)
 *
 * Packed layout: nq_pack_* rewrites the canonical codes and scales into two kernel-friendly
 * buffers, the packed codes Wq and the packed scales S: both are cut into tiles of 16 output
 * rows x one 64-wide K group, stored row-tile-major and contiguous along K; inside a tile the
 * codes are in the order of the tensor-core MMA operand fragments and the 16 scales in the
 * order the fragments' rows use them. Sizes depend only on (bits, K, N) and are exactly the
 * code bytes (nq_packed_bytes_*) and the scale bytes (nq_scale_bytes): no padding, no header.
 * The projection calls take the packed pair (Wq, S); the pages name neither layout, so both
 * are this library's definition.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers on the current CUDA device, owned by the caller; the
 *     library never frees or retains them. `stream` is a cudaStream_t (NULL = the legacy
 *     default stream). Calls are asynchronous on `stream`; none synchronises or prints.
 *   - Shapes: K % 64 == 0, N % 16 == 0, 0 <= T <= 64. T == 0 or N == 0 is an empty problem
 *     (NQ_OK, nothing launched). K == 0 makes Y an empty sum: zeros are written.
 *   - Token batches: one launch of the 8-token kernel handles up to 8 tokens (decode, and the
 *     T = 8 verify rounds the pages tune). An nq_gemm_q4/q5 or nq_swiglu_q4/q5 call with
 *     8 < T <= 64 (larger speculative-verify batches, e.g. 4 requests x 8 draft tokens) runs on
 *     the tensor-core kernel, which streams the weights once whatever T
 *     (nq_tensor_core_batches); so do nq_gemm_fp4 and nq_swiglu_fp4, and a grouped call runs
 *     one such launch per matrix. The no-allocation call with T > 8 runs one launch per slice of 8 tokens, each
 *     streaming the weights again, so its time grows with ceil(T / 8).
 *   - Alignment: every pointer 16-byte aligned.
 *   - All argument checks run on the host before anything is launched; a call that returns
 *     an error has launched nothing and left every output untouched.
 *   - Outputs must not overlap inputs (NQ_ERR_ALIAS).
 *   - The projection calls use a per-device workspace owned by the library (a few MB at
 *     most). It is allocated, or grown, on the first call that needs it: that call
 *     synchronises the device and must not be made during stream capture. nq_reserve
 *     allocates it ahead of time. Projection calls that overlap in time on one device
 *     (different streams, no ordering) share it and race: order them on one stream.
 *   - Device-side waits are bounded (2 s by default, see nq_wait_limit); a wait that runs
 *     out sets a device error flag that nq_device_error reads.
 *   - The projection calls (nq_gemm_*, nq_swiglu_*, the grouped calls) launch with programmatic
 *     dependent launch:
 *     their kernel may start while the previous kernel on `stream` is finishing. It reads
 *     X and writes Y, H and its workspace only after that kernel has completed, but starts
 *     streaming the packed weights at once: the weights must not be written by a kernel
 *     that lets its dependents start before its writes are done (one that calls
 *     cudaTriggerProgrammaticLaunchCompletion early). The environment variable NQ_PDL=0,
 *     read at the first call, turns this launch mode off.
 */
#ifndef NQ_H
#define NQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int nq_status;

enum {
    NQ_OK = 0,
    NQ_ERR_NULL = -1,     /* a required pointer is NULL                                   */
    NQ_ERR_SHAPE = -2,    /* K % 64, N % 16, T outside [0, 64], negative size, too large  */
    NQ_ERR_ALIGN = -3,    /* a pointer is not 16-byte aligned                             */
    NQ_ERR_ALIAS = -4,    /* an output range overlaps an input range                      */
    NQ_ERR_CUDA = -5,     /* a CUDA runtime call or kernel launch failed                  */
    NQ_ERR_DEVICE = -6,   /* current device is not compute capability 10.3 (sm_103)      */
    NQ_ERR_TIMEOUT = -7,  /* a bounded device-side wait ran out (reported by nq_device_error) */
    NQ_ERR_SCRATCH = -8   /* the problem needs more scratch than nq_gemm_q4_noalloc's fixed array */
};

/* Human-readable name of a status code. Never NULL; static storage. */
const char* nq_status_string(nq_status status);

/* Library version, (major << 16) | minor. */
int nq_version(void);

/* ---------------------------------------------------------------- packed sizes */

/* Bytes of the packed Q4 codes Wq: K*N/2. 0 on a bad shape (K % 64 or N % 16 nonzero). */
size_t nq_packed_bytes_q4(int K, int N);
/* Bytes of the packed Q5 codes Wq (nibble plane and high plane): 5*K*N/8. 0 on a bad shape. */
size_t nq_packed_bytes_q5(int K, int N);
/* Bytes of the packed scales S (Q4 or Q5): 2*N*(K/64), the same as the canonical scales. */
size_t nq_scale_bytes(int K, int N);

/* ---------------------------------------------------------------- offline repack */

/*
 * nq_pack_q4: canonical Q4 codes and scales -> packed pair (one-off "offline repack").
 *   wq_canon   device uint32 [N][K/8]     canonical codes
 *   s_canon    device fp16   [N][K/64]    canonical scales (bit patterns)
 *   wq_packed  device, nq_packed_bytes_q4(K, N) bytes, written (packed codes)
 *   s_packed   device, nq_scale_bytes(K, N) bytes, written (packed scales)
 * Pure bit permutation: nq_dequant_q4_debug(wq_packed, s_packed) reproduces the canonical
 * weights. Outputs must not overlap the inputs or each other (NQ_ERR_ALIAS).
 */
nq_status nq_pack_q4(const uint32_t* wq_canon, const uint16_t* s_canon, int K, int N, void* wq_packed,
                     void* s_packed, void* stream);

/* nq_pack_q5: as nq_pack_q4 for 5-bit codes given as nibble plane wn_canon [N][K/8] and
 * high plane wh_canon [N][K/32]; wq_packed holds nq_packed_bytes_q5(K, N) bytes. */
nq_status nq_pack_q5(const uint32_t* wn_canon, const uint32_t* wh_canon, const uint16_t* s_canon,
                     int K, int N, void* wq_packed, void* s_packed, void* stream);

/* ---------------------------------------------------------------- projections */

/*
 * nq_gemm_q4: Y = X * dequant(Wq, S) for 4-bit codes, 1 <= T <= 64 tokens.
 *   X   device bf16 [T][K]
 *   Wq  device packed codes, S device packed fp16 scales (both from nq_pack_q4)
 *   Y   device bf16 [T][N], written
 * Accumulation is fp32; Y is rounded once to bf16. Results are deterministic for a given
 * device (the split of K across thread blocks depends only on shape and SM count).
 */
nq_status nq_gemm_q4(const void* X, const void* Wq, const void* S, void* Y, int T, int K, int N,
                     void* stream);

/*
 * nq_gemm_q4_noalloc: nq_gemm_q4 for callers that cannot allocate device memory. The pages
 * have no counterpart; this is a library convenience.
 *
 * nq_gemm_q4 allocates its split-K scratch with cudaMalloc the first time a shape needs it.
 * Plug-ins whose host framework owns all device memory, and processes that must stay within
 * a fixed memory budget once serving has started (where a late allocation can fail, or
 * stall the device while it synchronises), cannot allow that. This call computes the
 * same Y with the same kernel but keeps its scratch in a fixed array of about 2.1 MB that
 * the library holds in every device's memory until the process exits; it calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   Arguments, layouts, alignment and results: as nq_gemm_q4.
 *   Limit: the call's work split needs S*ceil(N/32) + P <= 2048 partial slots and
 *   ceil(N/32) <= 4096 tickets, where S is the number of K slabs and P the number of thread
 *   blocks (nq_plan_info out[2] and out[0]; P <= the SM count). K fits one slab up to
 *   K = 49152 at T = 1, 24576 at T = 2, 16384 at T = 3, 12288 at T = 4, 8192 at T = 5..6 and
 *   6144 at T = 7..8; there, on a 152-SM GB300, N may be up to 60672. Each further slab
 *   divides the room: e.g. T = 8, K = 17408 (three slabs) allows N <= 20224. Larger
 *   problems return NQ_ERR_SCRATCH before anything is launched.
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *   with that device current; later calls on that device reuse it.
 *   Every call clears the tickets it uses on its own stream, then launches. All calls share
 *   the one array: calls that overlap on the GPU (unordered streams) race and give wrong
 *   results; order them on one stream.
 *   A bounded wait that runs out inside this call's kernel sets the array's own error word;
 *   it stays set until nq_device_error reports it (as NQ_ERR_TIMEOUT) and clears it.
 */
nq_status nq_gemm_q4_noalloc(const void* X, const void* Wq, const void* S, void* Y, int T, int K, int N,
                             void* stream);

/* nq_gemm_q5: as nq_gemm_q4 for 5-bit codes packed by nq_pack_q5 (z = 16). */
nq_status nq_gemm_q5(const void* X, const void* Wq, const void* S, void* Y, int T, int K, int N,
                     void* stream);

/*
 * Grouped projections: several matrices applied to the same X in one launch (e.g. the
 * attention q-gate 5120 x 6144 and kv 5120 x 1024 projections of a layer, which read the same
 * activations). One launch per 8-token slice carries all groups, so the per-launch start-up
 * and tail are paid once instead of once per matrix. No counterpart call on the pages, which
 * rely on CUDA graphs to chain a layer's launches ("NInfer-4090" post / NInfer digest,
 * decode with CUDA Graphs); this is the launch-level part of fusing a layer.
 */
typedef struct nq_group {
    const void* Wq;  /* packed codes of a K x N matrix (nq_pack_q4 / nq_pack_q5)            */
    const void* S;   /* its packed scales                                                  */
    void* Y;         /* bf16 [T][N] output, written                                        */
    int N;           /* outputs of this group: N % 16 == 0, N > 0                          */
} nq_group;

/*
 * nq_gemm_q4_grouped / nq_gemm_q5_grouped: Y_g = X * dequant(Wq_g, S_g) for each of `count`
 * groups (1..4, host array), all with the same X (device bf16 [T][K]) and code width.
 * Results equal those of one nq_gemm_q4 / nq_gemm_q5 call per group. T <= 8: one launch for
 * all groups; 8 < T <= 64 (tensor-core batches on): one tensor-core launch per group, each
 * streaming its weights once. Outputs must not overlap X, any group's weights or each other;
 * every argument is checked before the first launch. Errors as nq_gemm_q4.
 */
nq_status nq_gemm_q4_grouped(const void* X, const nq_group* groups, int count, int T, int K, void* stream);
nq_status nq_gemm_q5_grouped(const void* X, const nq_group* groups, int count, int T, int K, void* stream);

/*
 * nq_swiglu_q4: fused gate/up projection of the SwiGLU MLP ("NInfer-4090" release post,
 * section "V3 做了什么", SwiGLU path at T=8):
 *   g = X * dequant(Wg, Sg),  u = X * dequant(Wu, Su)   (each [T][N], fp32 accumulation)
 *   H = bf16(silu(g) * u),    silu(g) = g / (1 + exp(-g)) in fp32
 *   X device bf16 [T][K]; (Wg, Sg) and (Wu, Su) packed by nq_pack_q4 (K x N each);
 *   H device bf16 [T][N], written. The down projection is nq_gemm_q4 on H.
 * T <= 8: one launch that computes g and u together. 8 < T <= 64 (with tensor-core batches
 * on): two launches of the tensor-core kernel on the same X, the gate projection writing g in
 * fp32 to a library buffer (T x N floats, see nq_reserve) and the up projection finishing
 * H = bf16(silu(g) * u) from it; the same fp32 arithmetic, each weight matrix streamed once.
 */
nq_status nq_swiglu_q4(const void* X, const void* Wg, const void* Sg, const void* Wu, const void* Su,
                       void* H, int T, int K, int N, void* stream);

/*
 * nq_swiglu_q5: as nq_swiglu_q4 for 5-bit gate and up weights packed by nq_pack_q5
 * (z = 16): the pages run the SwiGLU path among the small-batch Q4/Q5 projections
 * ("NInfer-4090" release post, section "V3 做了什么"; "ninfer-ext" README, the Q5
 * small-batch path). Same arguments, layouts, ownership and errors; the down projection is
 * nq_gemm_q4 or nq_gemm_q5 on H.
 */
nq_status nq_swiglu_q5(const void* X, const void* Wg, const void* Sg, const void* Wu, const void* Su,
                       void* H, int T, int K, int N, void* stream);

/* ---------------------------------------------------------------- NVFP4 weights */

/*
 * NVFP4 weights: the 4-bit floating-point format the pages run beside groupwise int
 * ("ninfer-ext" README, section "与原版 NInfer 的对比": an NVFP4 MLP-projection tensor-core
 * kernel with 16-bit activations, "A16"). The pages print no layout; this library reads NVFP4
 * as: e2m1 elements (sign, 2 exponent bits with bias 1, 1 mantissa bit; values 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6 and their negatives), one e4m3 scale (bias 7, the "fn" variant) per 16
 * consecutive elements along K, and one fp32 tensor scale g:
 *     W[k,n] = g * e4m3(sf[n, k/16]) * e2m1(c[n,k]),   Y[t,n] = sum_k X[t,k] * W[k,n].
 * Canonical layouts: codes uint32 [N][K/8], nibble i of word j the code of k = 8j+i (the Q4
 * rule); scales uint8 [N][K/16] e4m3 bit patterns. K % 64 == 0, N % 16 == 0 as above.
 * The kernels decode each weight pair into fp16 exactly (scale times element has at most 6
 * significant bits) and run fp16 tensor-core MMAs against X converted to fp16 with a
 * per-token power-of-two range factor; accumulation is fp32, Y is rounded once to bf16.
 */

/* Bytes of packed NVFP4 codes (K*N/2) and of packed NVFP4 block scales (N*K/16). */
size_t nq_packed_bytes_fp4(int K, int N);
size_t nq_scale_bytes_fp4(int K, int N);

/* nq_pack_fp4: canonical NVFP4 codes and e4m3 scales (device) -> packed pair (device, sizes
 * above); outputs must not overlap the inputs or each other. */
nq_status nq_pack_fp4(const uint32_t* codes_canon, const uint8_t* sf_canon, int K, int N, void* wq_packed,
                      void* s_packed, void* stream);

/* nq_gemm_fp4: Y = X * W for NVFP4 weights packed by nq_pack_fp4, global_scale = g,
 * 1 <= T <= 64 (8 < T <= 64 on the tensor-core kernel as the other projections: the decoded
 * weights e2m1 x e4m3 are exact in bf16). Arguments, alignment, errors and launch behaviour as
 * nq_gemm_q4. */
nq_status nq_gemm_fp4(const void* X, const void* Wq, const void* S, float global_scale, void* Y, int T, int K,
                      int N, void* stream);

/*
 * nq_swiglu_fp4: the SwiGLU block of an NVFP4 MLP (the pages' NVFP4 MLP projections, "ninfer-ext"
 * README, section "与原版 NInfer 的对比"): as nq_swiglu_q4 with gate and up weights packed by
 * nq_pack_fp4, each with its own tensor scale:
 *   g = X * W(Wg, Sg, gate_scale),  u = X * W(Wu, Su, up_scale),  H = bf16(silu(g) * u).
 * T <= 8: one launch computing g and u together (fp16 operands, tensor scales applied to the
 * fp32 partials); 8 < T <= 64: the two tensor-core launches of nq_swiglu_q4. Arguments,
 * alignment, errors and launch behaviour as nq_swiglu_q4; the down projection is nq_gemm_fp4
 * on H.
 */
nq_status nq_swiglu_fp4(const void* X, const void* Wg, const void* Sg, float gate_scale, const void* Wu,
                        const void* Su, float up_scale, void* H, int T, int K, int N, void* stream);

/* nq_dequant_fp4_debug: out[n][k] = g * (scale * element) in fp32 through the kernels' own
 * decoder; exact, so it must equal the CPU definition bit for bit. */
nq_status nq_dequant_fp4_debug(const void* Wq, const void* S, float global_scale, float* out, int K, int N,
                               void* stream);

/* ---------------------------------------------------------------- debug dumps */

/*
 * nq_dequant_q4_debug: decodes the PACKED pair (Wq, S) with the decoder of the T <= 2
 * projection kernels (fp16 operands: a code q becomes 1024 + q, or 1024 + 16 q at the upper
 * half of each 16-wide K step) and writes out[n][k] = (float)s * (float)(q - 8) in fp32,
 * canonical order [N][K]. The value is exact, so it must equal the CPU definition bit for bit.
 */
nq_status nq_dequant_q4_debug(const void* Wq, const void* S, float* out, int K, int N, void* stream);

/* nq_dequant_q5_debug: as above for a Q5 packed pair (z = 16). */
nq_status nq_dequant_q5_debug(const void* Wq, const void* S, float* out, int K, int N, void* stream);

/*
 * nq_dequant_q4_debug_bf16 / nq_dequant_q5_debug_bf16: the same dump through the decoder of
 * the T >= 3 projection kernels (bf16 operands: every code q becomes 128 + q). Same
 * arguments and result; the two decoders must agree with each other and with the CPU
 * definition bit for bit.
 */
nq_status nq_dequant_q4_debug_bf16(const void* Wq, const void* S, float* out, int K, int N, void* stream);
nq_status nq_dequant_q5_debug_bf16(const void* Wq, const void* S, float* out, int K, int N, void* stream);

/* ---------------------------------------------------------------- recorded programs */

/*
 * A program: a sequence of projection calls (a decoder layer, or a stack of layers) recorded
 * once and replayed as one CUDA graph. The pages run decode through CUDA graphs ("ninfer-ext"
 * README, section "推荐设置": keep CUDA graphs on; NInfer digest, section "项目定位": the
 * engine uses CUDA graphs in the decode phase; "NInfer-4090" post, section "快速启动": the
 * graphs are built once at start-up, outside the steady-state decode time). A program is that
 * step for this library's calls: every launch of every recorded call is captured in the
 * recorded order, with the work split, tensor maps and workspace addresses fixed at build
 * time, and nq_program_launch then costs one graph launch instead of one host call per kernel.
 *
 * What a program fixes and what it does not:
 *   - It records the DEVICE ADDRESSES of X, the packed weights and the outputs, not their
 *     contents: a launch reads whatever X holds at that point (write the next token's
 *     activations into the same buffer, then launch again). The buffers must stay allocated
 *     while the program can be launched; the library never frees them.
 *   - Shapes (T, K, N) are fixed; a different token count needs another program.
 *   - The library settings in force at build time are baked in: tensor-core batches
 *     (nq_tensor_core_batches), slab clusters, the wait bound (nq_wait_limit) and the
 *     dependent-launch mode.
 *   - The per-device workspace addresses are baked in as well. nq_program_build reserves the
 *     workspace for every recorded call first (as nq_reserve), so that capture allocates
 *     nothing. If the workspace is later reallocated (a larger call or nq_reserve grew it,
 *     or nq_shutdown freed it), the next nq_program_launch builds the program again before
 *     launching it (nq_program_info counts the builds).
 *   - A program belongs to the device that was current when it was built; launching it with
 *     another current device returns NQ_ERR_DEVICE.
 *   - One program must not be used by several host threads at once. Programs, like the
 *     projection calls themselves, share the device workspace: launches that overlap in time
 *     (different streams, no ordering) race. Order them on one stream.
 *
 * Results are those of making the recorded calls, in order, on one stream: the kernels are
 * deterministic, so a replay writes the same bits as the eager calls.
 */
typedef struct nq_program nq_program;

/* nq_program_create: a new, empty program in *out (host memory only; no CUDA call).
 * NQ_ERR_NULL if out is NULL; NQ_ERR_CUDA if the host allocation fails. */
nq_status nq_program_create(nq_program** out);

/*
 * Recording calls: append one projection call to the program. Arguments, layouts and
 * ownership are those of the call named (nq_gemm_q4 / nq_gemm_q5 for bits 4 / 5,
 * nq_gemm_fp4, nq_swiglu_q4 / nq_swiglu_q5, nq_swiglu_fp4, nq_gemm_q4_grouped /
 * nq_gemm_q5_grouped), without
 * the stream. Every host-side check of that call runs here, on the host and without a GPU
 * (shape, NULL, alignment, aliasing: the same status codes); a call that fails them is not
 * recorded. An empty call (T == 0 or N == 0) is accepted and records nothing. Recording into
 * a program that was built marks it for building again. The grouped call copies `groups`.
 */
nq_status nq_program_gemm(nq_program* prog, int bits, const void* X, const void* Wq, const void* S, void* Y, int T,
                          int K, int N);
nq_status nq_program_gemm_fp4(nq_program* prog, const void* X, const void* Wq, const void* S, float global_scale,
                              void* Y, int T, int K, int N);
nq_status nq_program_swiglu(nq_program* prog, int bits, const void* X, const void* Wg, const void* Sg,
                            const void* Wu, const void* Su, void* H, int T, int K, int N);
nq_status nq_program_swiglu_fp4(nq_program* prog, const void* X, const void* Wg, const void* Sg, float gate_scale,
                                const void* Wu, const void* Su, float up_scale, void* H, int T, int K, int N);
nq_status nq_program_grouped(nq_program* prog, int bits, const void* X, const nq_group* groups, int count, int T,
                             int K);

/*
 * nq_program_build: reserve the current device's workspace for every recorded call, capture
 * the calls in order into a CUDA graph (on a stream the program owns) and instantiate it.
 * Synchronises the device when the workspace has to grow. On an error from a recorded call
 * the capture is abandoned, nothing has run, and that status is returned (nq_program_info
 * names the call). A program with no recorded calls builds to an empty graph.
 */
nq_status nq_program_build(nq_program* prog);

/*
 * nq_program_launch: launch the program's graph on `stream` (a cudaStream_t; NULL = the
 * legacy default stream), asynchronously, building it first if it has not been built or the
 * workspace has moved since. Errors: NQ_ERR_NULL, NQ_ERR_DEVICE (another device is current),
 * a build error, NQ_ERR_CUDA. A bounded device-side wait that runs out is reported by
 * nq_device_error, as for the eager calls.
 */
nq_status nq_program_launch(nq_program* prog, void* stream);

/*
 * nq_program_info: out[0] recorded calls, out[1] kernel launches in the built graph (0 if not
 * built), out[2] builds so far, out[3] index of the recorded call whose error ended the last
 * build, or -1. No GPU needed.
 */
nq_status nq_program_info(const nq_program* prog, int64_t out[4]);

/* nq_program_destroy: free the program's graph, its stream and its records. Does not
 * synchronise: a launch still in flight completes, and its graph is freed after it. NULL is
 * ignored. The recorded buffers are untouched. */
void nq_program_destroy(nq_program* prog);

/* ---------------------------------------------------------------- runtime */

/*
 * nq_reserve: allocate the current device's workspace for projections of up to
 * (T_max, K_max, N_max) now, so that later calls of at most that size allocate nothing
 * (e.g. before capturing a CUDA graph). With T_max > 8 this includes the tensor-core
 * kernel's partial sums (at most max(SMs, N_max / 128) x 128 x 64 floats, about 5 MB) and
 * the fp32 gate outputs of its SwiGLU calls (T_max x N_max floats).
 * Synchronises the device.
 */
nq_status nq_reserve(int T_max, int K_max, int N_max);

/*
 * nq_device_error: synchronise the current device, then report and clear the device-side
 * error flags of its workspace and of nq_gemm_q4_noalloc's fixed scratch: NQ_OK, or
 * NQ_ERR_TIMEOUT if a bounded wait inside a kernel ran out since the last check (that
 * call's outputs are then undefined). Clears the split-K tickets as well, so later calls
 * start clean.
 */
nq_status nq_device_error(void);

/*
 * nq_wait_limit: the bound, in nanoseconds, of every device-side wait of later projection
 * calls (a pipeline stage, an activation slab, a cluster peer). ns > 0 sets it; ns <= 0 only
 * queries. Returns the previous bound. Default 2 s, or the environment variable NQ_WAIT_NS
 * read at the first call. A wait that runs out aborts its thread block (its outputs are
 * undefined, nq_device_error reports NQ_ERR_TIMEOUT) after the block has waited, on a
 * separate fixed bound, for the copies it already issued. A bound far below a kernel's run
 * time makes calls abort: that is how the tests reach this path.
 */
long long nq_wait_limit(long long ns);

/* nq_shutdown: free every device workspace of this process (synchronises each device). */
void nq_shutdown(void);

/*
 * nq_plan_info: the work split a projection of this shape would use, for inspection and
 * host-side tests (no GPU needed). mode 0 = gemm, 1 = swiglu. num_sms = SMs to plan for.
 *   out[0] ctas      thread blocks launched (persistent, at most one per SM)
 *   out[1] units     work units (one unit = two 16-row tiles x one 64-wide K group)
 *   out[2] slabs     K slabs (K is cut when T*K activations exceed the on-chip X buffer)
 *   out[3] slab_groups  64-wide groups per slab (the last slab may be shorter)
 *   out[4] pairs     row pairs (gemm: pairs of 16-row tiles; swiglu: gate/up tile pairs)
 *   out[5] ws_slots  fp32 partial-sum slots of the workspace used by this shape
 *   out[6] stages    shared-memory pipeline stages
 *   out[7] chunk_groups  K groups per pipeline stage
 */
nq_status nq_plan_info(int bits, int mode, int T, int K, int N, int num_sms, int64_t out[8]);

/*
 * nq_plan_segments: the (slab, pair, first group, end group) runs that thread block `cta`
 * processes, in order, for the same plan as nq_plan_info. Writes up to `cap` rows of 4
 * int64 into `seg`; returns the number of runs (which may exceed cap), or a negative status.
 */
int64_t nq_plan_segments(int bits, int mode, int T, int K, int N, int num_sms, int cta,
                         int64_t* seg, int64_t cap);

/*
 * nq_tensor_core_batches: how projections (Q4, Q5, NVFP4) and SwiGLU blocks with
 * 8 < T <= 64 run. On (1, the default; the environment variable NQ_TC=0 read at the first call
 * turns it off): one launch of the tensor-core kernel per weight matrix (two for a SwiGLU
 * block), which decodes the weights once into the fifth-generation tensor cores' memory (TMEM)
 * and multiplies them with all T tokens (tcgen05.mma, M = 128 rows, N = 16, 32 or 64 padded
 * tokens), so the weights stream from HBM once. Off (0): one launch of the 8-token kernel per
 * slice of 8 tokens. -1 only queries. Returns the previous setting. Either way the results
 * agree with the oracle within the same tolerance. A grouped call runs one such launch per
 * matrix. The no-allocation call uses slices at every T. Not synchronised with calls in
 * flight.
 */
int nq_tensor_core_batches(int enable);

/*
 * nq_plan_tc_info: the work split the tensor-core kernel would use (host only): out[0] blocks,
 * [1] row blocks of 128 rows, [2] K pieces per row block (their fp32 partials are added in
 * fixed order by the row block's last piece), [3] padded token count, [4] pipeline stages,
 * [5] shared-memory bytes, [6] 64-wide K groups, [7] groups per stage. bits 4, 5 or 14 (NVFP4
 * weights), 8 < T <= 64.
 */
nq_status nq_plan_tc_info(int bits, int T, int K, int N, int num_sms, int64_t out[8]);

/*
 * nq_route_info: which kernel and variant a projection call of this shape takes with the
 * current settings (nq_tensor_core_batches, nq_slab_clusters), for a GPU of num_sms SMs; host
 * only, no GPU needed. The pages route their small-batch projections by shape ("NInfer-4090"
 * release post, section "V3 做了什么": T=8 routing); this is the library's routing, each
 * choice measured on GB300. bits 4, 5 or 14 (NVFP4); mode 0 = gemm, 1 = SwiGLU block;
 * 1 <= T <= 64.
 *   out[0] kernel: 0 = the 8-token kernel (mma.sync), 1 = the tensor-core kernel (tcgen05)
 *   out[1] launches per call (slices of 8 tokens, or the SwiGLU block's two tensor-core launches)
 *   out[2] MMA operand type: 0 = fp16 (T <= 2, and NVFP4 on the 8-token kernel), 1 = bf16
 *   out[3] work split: 0 = stream-K over the SMs, 1 = whole row pairs per block, 2 = slab
 *          clusters, 3 = 128-row blocks times K pieces (tensor-core kernel)
 *   out[4] blocks of the (first) launch
 *   out[5] K slabs (8-token kernel) or K pieces per row block (tensor-core kernel)
 *   out[6] pipeline stages
 *   out[7] padded token count of the (first) launch
 * With slab clusters on, their plan assumes that all num_sms / S clusters can be resident.
 */
nq_status nq_route_info(int bits, int mode, int T, int K, int N, int num_sms, int64_t out[8]);

/*
 * nq_slab_clusters: turn slab clusters on (1) or off (0) for later projection calls of this
 * process, or only query (-1); returns the previous setting. Off unless the environment
 * variable NQ_CLUSTER is "1" at the first call. On GB300 a slab-cluster call is 8-23 %
 * faster than the stream-K one when such calls follow each other, but a slab-cluster launch
 * behind a different projection kernel under programmatic dependent launch started late
 * (with NQ_PDL=0 it was faster there too), so slab-cluster launches go without dependent
 * launch and the mode is opt-in. Not synchronised with calls in flight on other threads.
 */
int nq_slab_clusters(int enable);

/*
 * nq_plan_cluster_info / nq_plan_cluster_segments: the same for a slab-cluster launch,
 * which the projection calls use (bf16 operands, T >= 3) when K needs 2..4 slabs, enough
 * thread-block clusters fit the device, and slab clusters are on (nq_slab_clusters). A cluster of S blocks takes a range of (row pair, slab-local group)
 * work; block rank r takes slab r of it, stages that activation slab once, and the S parts
 * of each run are added on chip by rank 0 (distributed shared memory) before the usual
 * split-K settle between clusters. Host only; no device needed.
 *   clusters: clusters to plan for (the calls use the device's resident count, at most
 *   SMs / S).
 *   info out[8]: [0] blocks, [1] cluster size S, [2] groups per slab, [3] row pairs,
 *   [4] partial-sum slots, [5] pipeline stages, [6] cluster-level units, [7] clusters.
 *   segments: as nq_plan_segments for block `cta` (cluster cta / S, rank cta % S): its
 *   real (slab, pair, first group, end group) runs; a run may be empty (ga == gb) when the
 *   last slab is shorter. Returns NQ_ERR_SHAPE when the shape has no slab-cluster plan.
 */
nq_status nq_plan_cluster_info(int bits, int mode, int T, int K, int N, int clusters, int64_t out[8]);
int64_t nq_plan_cluster_segments(int bits, int mode, int T, int K, int N, int clusters, int cta,
                                 int64_t* seg, int64_t cap);

#ifdef __cplusplus
}
#endif

#endif /* NQ_H */
