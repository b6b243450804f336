/*
 * Plain CPU oracle for the weight-only groupwise int4/int5 projection.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, the package's smoke check and the bench's
 * CPU-baseline leg may load this. It shares no code, header, table or constant with
 * the CUDA library, and never sees the packed (kernel) layout: it reads the canonical
 * layout directly.
 *
 * What it computes (the projection the pages tune for small batches:
 * "NInfer-4090" release post, section "V3 做了什么" -- small-batch Q4/Q5 projections,
 * T=8 routing, GDN and attention projections and the SwiGLU path; "ninfer-ext"
 * README, section "与原版 NInfer 的对比" -- the Q5 small-batch path for speculative
 * verify rounds):
 *
 *   Y[t,n] = sum_k X[t,k] * W[k,n],  W[k,n] = s[n, k/64] * (q[n,k] - z),
 *   z = 8 for 4-bit codes, z = 16 for 5-bit codes.
 *
 * The pages do not print the format; the layout below is this library's definition:
 *   Q4: Wq uint32 [N][K/8], nibble i of word j is q[n, 8j+i] (low nibble first)
 *   Q5: Wn uint32 [N][K/8] (low 4 bits, same rule) and Wh uint32 [N][K/32],
 *       bit i of word j is bit 4 of q[n, 32j+i]; q = nib | hi << 4
 *   S : fp16 [N][K/64];  X: bf16 [T][K];  Y: [T][N]
 *
 * Precision: the dequantised weight is formed as ONE fp32 multiply,
 * (float)s * (float)(q - z). It is exact: |q - z| <= 16 needs 5 bits and an fp16
 * significand has 11, so the product fits in fp32's 24. The contraction is summed in
 * fp64 in increasing k. SwiGLU: g and u in fp64, h = silu(g) * u in fp64, then
 * rounded once to bf16 (round to nearest, ties to even).
 *
 * Each exported function says which of the steps above it implements.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, written from the format definition:
 * sign 1 bit, exponent 5 bits (bias 15), fraction 10 bits.
 * exponent 0: subnormal, value = fraction * 2^-24; exponent 31: inf / NaN. */
double orc_fp16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32: widen by appending 16 zero bits. */
double orc_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> bf16, round to nearest, ties to even, from the format definition:
 * 8 significant bits for normal numbers (exponent >= -126), a fixed quantum of 2^-133
 * below that; overflow past the largest finite value rounds to infinity. */
uint16_t orc_round_bf16(double v) {
    if (isnan(v)) return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a = m * 2^e, 0.5 <= m < 1 */
    int q_exp = (e - 1 >= -126) ? (e - 1 - 7) : (-126 - 7);
    double quantum = ldexp(1.0, q_exp);
    double r = nearbyint(a / quantum) * quantum; /* default rounding mode: ties to even */
    const double max_bf16 = ldexp(255.0, 127 - 7);  /* (2 - 2^-7) * 2^127 */
    if (r > max_bf16) return sign | 0x7f80;
    /* r is exactly representable: read its bits through binary32. */
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7fff);
}

/* Canonical unpack: 4-bit code q[n,k]. */
static inline int q4_code(const uint32_t* wq, int K, int n, int k) {
    uint32_t word = wq[(size_t)n * (K / 8) + (k >> 3)];
    return (int)((word >> (4 * (k & 7))) & 0xFu);
}

/* Canonical unpack: 5-bit code q[n,k] = nibble | high bit << 4. */
static inline int q5_code(const uint32_t* wn, const uint32_t* wh, int K, int n, int k) {
    uint32_t nw = wn[(size_t)n * (K / 8) + (k >> 3)];
    uint32_t hw = wh[(size_t)n * (K / 32) + (k >> 5)];
    int nib = (int)((nw >> (4 * (k & 7))) & 0xFu);
    int hi = (int)((hw >> (k & 31)) & 1u);
    return nib | (hi << 4);
}

/* Dequantised weight in fp32: one multiply of the fp16 scale by the integer (q - z). */
static inline float dequant(const uint16_t* s, int K, int n, int k, int q, int z) {
    float scale = (float)orc_fp16_to_f64(s[(size_t)n * (K / 64) + (k >> 6)]);
    return scale * (float)(q - z);
}

/* Step "dequantise": W32[n][k] for the 4-bit format (row n = output feature). */
void orc_dequant_q4(const uint32_t* wq, const uint16_t* s, int K, int N, float* w) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            w[(size_t)n * K + k] = dequant(s, K, n, k, q4_code(wq, K, n, k), 8);
}

/* Step "dequantise": W32[n][k] for the 5-bit format. */
void orc_dequant_q5(const uint32_t* wn, const uint32_t* wh, const uint16_t* s, int K, int N,
                    float* w) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            w[(size_t)n * K + k] = dequant(s, K, n, k, q5_code(wn, wh, K, n, k), 16);
}

/* Steps "dequantise" + "contract" for one output row n, all T tokens, fp64 in k order. */
static void row_q4(const uint16_t* x, const uint32_t* wq, const uint16_t* s, int T, int K, int n,
                   float* wrow, double* out /* [T] */) {
    for (int k = 0; k < K; ++k) wrow[k] = dequant(s, K, n, k, q4_code(wq, K, n, k), 8);
    for (int t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += (double)wrow[k] * orc_bf16_to_f64(x[(size_t)t * K + k]);
        out[t] = acc;
    }
}

static void row_q5(const uint16_t* x, const uint32_t* wn, const uint32_t* wh, const uint16_t* s,
                   int T, int K, int n, float* wrow, double* out) {
    for (int k = 0; k < K; ++k) wrow[k] = dequant(s, K, n, k, q5_code(wn, wh, K, n, k), 16);
    for (int t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += (double)wrow[k] * orc_bf16_to_f64(x[(size_t)t * K + k]);
        out[t] = acc;
    }
}

/* Y[t][n] in fp64 for the 4-bit format (rows parallelised over n). */
void orc_gemm_q4(const uint16_t* x, const uint32_t* wq, const uint16_t* s, int T, int K, int N,
                 double* y) {
#pragma omp parallel
    {
        float* wrow = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
        double* out = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(static)
        for (int n = 0; n < N; ++n) {
            row_q4(x, wq, s, T, K, n, wrow, out);
            for (int t = 0; t < T; ++t) y[(size_t)t * N + n] = out[t];
        }
        free(out);
        free(wrow);
    }
}

/* Y[t][n] in fp64 for the 5-bit format. */
void orc_gemm_q5(const uint16_t* x, const uint32_t* wn, const uint32_t* wh, const uint16_t* s,
                 int T, int K, int N, double* y) {
#pragma omp parallel
    {
        float* wrow = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
        double* out = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(static)
        for (int n = 0; n < N; ++n) {
            row_q5(x, wn, wh, s, T, K, n, wrow, out);
            for (int t = 0; t < T; ++t) y[(size_t)t * N + n] = out[t];
        }
        free(out);
        free(wrow);
    }
}

/* Selected rows only: y[i][t] for n = rows[i], all T tokens (for full-size spot checks). */
void orc_gemm_q4_rows(const uint16_t* x, const uint32_t* wq, const uint16_t* s, int T, int K,
                      const int* rows, int count, double* y /* [count][T] */) {
#pragma omp parallel
    {
        float* wrow = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic)
        for (int i = 0; i < count; ++i) row_q4(x, wq, s, T, K, rows[i], wrow, y + (size_t)i * T);
        free(wrow);
    }
}

void orc_gemm_q5_rows(const uint16_t* x, const uint32_t* wn, const uint32_t* wh,
                      const uint16_t* s, int T, int K, const int* rows, int count, double* y) {
#pragma omp parallel
    {
        float* wrow = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic)
        for (int i = 0; i < count; ++i)
            row_q5(x, wn, wh, s, T, K, rows[i], wrow, y + (size_t)i * T);
        free(wrow);
    }
}

/* SwiGLU epilogue in fp64: silu(g) * u with silu(g) = g / (1 + e^-g). */
double orc_silu_mul(double g, double u) { return g / (1.0 + exp(-g)) * u; }

/* Fused gate/up block: G, U in fp64 ([T][N] each) and H = bf16(silu(G) * U) ([T][N]). */
void orc_swiglu_q4(const uint16_t* x, const uint32_t* wg, const uint16_t* sg,
                   const uint32_t* wu, const uint16_t* su, int T, int K, int N, double* g,
                   double* u, uint16_t* h) {
    orc_gemm_q4(x, wg, sg, T, K, N, g);
    orc_gemm_q4(x, wu, su, T, K, N, u);
    for (size_t i = 0; i < (size_t)T * N; ++i) h[i] = orc_round_bf16(orc_silu_mul(g[i], u[i]));
}

/* Same block on selected rows: g, u, h are [count][T]. */
void orc_swiglu_q4_rows(const uint16_t* x, const uint32_t* wg, const uint16_t* sg,
                        const uint32_t* wu, const uint16_t* su, int T, int K, const int* rows,
                        int count, double* g, double* u, uint16_t* h) {
    orc_gemm_q4_rows(x, wg, sg, T, K, rows, count, g);
    orc_gemm_q4_rows(x, wu, su, T, K, rows, count, u);
    for (size_t i = 0; i < (size_t)count * T; ++i) h[i] = orc_round_bf16(orc_silu_mul(g[i], u[i]));
}

/* The same block for 5-bit gate and up weights (nibble plane + high plane each, z = 16). */
void orc_swiglu_q5(const uint16_t* x, const uint32_t* wgn, const uint32_t* wgh, const uint16_t* sg,
                   const uint32_t* wun, const uint32_t* wuh, const uint16_t* su, int T, int K, int N,
                   double* g, double* u, uint16_t* h) {
    orc_gemm_q5(x, wgn, wgh, sg, T, K, N, g);
    orc_gemm_q5(x, wun, wuh, su, T, K, N, u);
    for (size_t i = 0; i < (size_t)T * N; ++i) h[i] = orc_round_bf16(orc_silu_mul(g[i], u[i]));
}

void orc_swiglu_q5_rows(const uint16_t* x, const uint32_t* wgn, const uint32_t* wgh,
                        const uint16_t* sg, const uint32_t* wun, const uint32_t* wuh,
                        const uint16_t* su, int T, int K, const int* rows, int count, double* g,
                        double* u, uint16_t* h) {
    orc_gemm_q5_rows(x, wgn, wgh, sg, T, K, rows, count, g);
    orc_gemm_q5_rows(x, wun, wuh, su, T, K, rows, count, u);
    for (size_t i = 0; i < (size_t)count * T; ++i) h[i] = orc_round_bf16(orc_silu_mul(g[i], u[i]));
}

/* ---------------------------------------------------------------- NVFP4 weights
 *
 * The 4-bit floating-point weight format the pages name beside groupwise int ("ninfer-ext"
 * README, section "与原版 NInfer 的对比": the NVFP4 MLP-projection A16 tensor-core kernel).
 * The pages print no layout; the plain reading of NVFP4 is used:
 *   element  e2m1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0;
 *            exponent 0 is subnormal: value = m * 0.5; otherwise 2^(e-1) * (1 + m/2)
 *   block    16 consecutive elements along K share one scale,
 *   scale    e4m3 (the "fn" variant): sign bit 7, exponent bits 6..3 (bias 7), mantissa
 *            bits 2..0; exponent 0 is subnormal: m * 2^-9; S.1111.111 is NaN; no infinity
 *   tensor   one fp32 scale g for the whole matrix
 *   W[n,k] = g * scale(sf[n, k/16]) * e2m1(c[n,k]),  Y[t,n] = sum_k X[t,k] * W[n,k]
 * Canonical layout: codes uint32 [N][K/8] with nibble i of word j the code of k = 8j+i (the
 * same rule as the 4-bit integer codes), scales uint8 [N][K/16] e4m3 bit patterns.
 * Dequantised weight in fp32: (float)g * (float)(scale * element); the inner product is
 * exact in fp32 (at most 2 + 4 significant bits), so it is rounded once. */

double orc_e2m1_to_f64(uint8_t c) {
    int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

double orc_e4m3_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);           /* m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

static inline float fp4_weight(const uint32_t* codes, const uint8_t* sf, float g, int K, int n, int k) {
    uint8_t c = (uint8_t)q4_code(codes, K, n, k);
    float inner = (float)(orc_e4m3_to_f64(sf[(size_t)n * (K / 16) + (k >> 4)]) * orc_e2m1_to_f64(c));
    return g * inner;
}

/* Step "dequantise" for NVFP4: W32[n][k]. */
void orc_dequant_fp4(const uint32_t* codes, const uint8_t* sf, float g, int K, int N, float* w) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) w[(size_t)n * K + k] = fp4_weight(codes, sf, g, K, n, k);
}

static void row_fp4(const uint16_t* x, const uint32_t* codes, const uint8_t* sf, float g, int T, int K, int n,
                    float* wrow, double* out) {
    for (int k = 0; k < K; ++k) wrow[k] = fp4_weight(codes, sf, g, K, n, k);
    for (int t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += (double)wrow[k] * orc_bf16_to_f64(x[(size_t)t * K + k]);
        out[t] = acc;
    }
}

/* Y[t][n] in fp64 for NVFP4 weights (dequantise + contract, k order). */
void orc_gemm_fp4(const uint16_t* x, const uint32_t* codes, const uint8_t* sf, float g, int T, int K, int N,
                  double* y) {
#pragma omp parallel
    {
        float* wrow = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
        double* out = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(static)
        for (int n = 0; n < N; ++n) {
            row_fp4(x, codes, sf, g, T, K, n, wrow, out);
            for (int t = 0; t < T; ++t) y[(size_t)t * N + n] = out[t];
        }
        free(out);
        free(wrow);
    }
}

void orc_gemm_fp4_rows(const uint16_t* x, const uint32_t* codes, const uint8_t* sf, float g, int T, int K,
                       const int* rows, int count, double* y /* [count][T] */) {
#pragma omp parallel
    {
        float* wrow = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic)
        for (int i = 0; i < count; ++i) row_fp4(x, codes, sf, g, T, K, rows[i], wrow, y + (size_t)i * T);
        free(wrow);
    }
}

/* The SwiGLU block of an NVFP4 MLP: gate and up matrices, each with its own tensor scale;
 * G, U in fp64 ([T][N] each) and H = bf16(silu(G) * U). */
void orc_swiglu_fp4(const uint16_t* x, const uint32_t* cg, const uint8_t* sfg, float gg, const uint32_t* cu,
                    const uint8_t* sfu, float gu, int T, int K, int N, double* g, double* u, uint16_t* h) {
    orc_gemm_fp4(x, cg, sfg, gg, T, K, N, g);
    orc_gemm_fp4(x, cu, sfu, gu, T, K, N, u);
    for (size_t i = 0; i < (size_t)T * N; ++i) h[i] = orc_round_bf16(orc_silu_mul(g[i], u[i]));
}

void orc_swiglu_fp4_rows(const uint16_t* x, const uint32_t* cg, const uint8_t* sfg, float gg, const uint32_t* cu,
                         const uint8_t* sfu, float gu, int T, int K, const int* rows, int count, double* g,
                         double* u, uint16_t* h) {
    orc_gemm_fp4_rows(x, cg, sfg, gg, T, K, rows, count, g);
    orc_gemm_fp4_rows(x, cu, sfu, gu, T, K, rows, count, u);
    for (size_t i = 0; i < (size_t)count * T; ++i) h[i] = orc_round_bf16(orc_silu_mul(g[i], u[i]));
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
