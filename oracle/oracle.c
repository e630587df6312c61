/*
 * oracle.c — plain CPU reference for the tiled GEMM D = A·Bᵀ.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library
 * is checked against.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the library under tiled_mma_atom_gb300/; the library never calls it.
 *
 * What it computes (all sums in fp64, k in increasing order, no blocking):
 *
 *   D[m,n] = sum_{k<K} a(m,k) * b(n,k)
 *
 * - Operand convention A = (M,K), B = (N,K), D = (M,N): "add-target-atom-op",
 *   §1.4 (ThrVal layouts: reference tiles (M,K) for A, (N,K) for B, (M,N)
 *   for C) and §1.5.3 (reference coordinate system).
 * - a(m,k) = decode(A[crd2idx((m,k), layoutA)]) with crd2idx the sum of
 *   coordinate times stride: "FlyDSL Kernel Authoring Skill", §2 Layout
 *   System, "Coordinate Mapping" (formula and worked example).
 * - A coordinate that indexes a nested mode (for example the second mode of
 *   (9,(4,8))) is split colexicographically, first sub-mode fastest — the
 *   same order that idx2crd uses in the worked example of "Coordinate
 *   Mapping" (43 -> (43 % 8, 43 / 8)); nested shapes appear under
 *   "Construction" in the same section.
 * - MXFP4: one E8M0 scale per 32 consecutive K-elements: "FlyDSL Kernel
 *   Authoring Skill", §6 MFMA Integration, "gfx1250 WMMA (wave32)",
 *   MX-scaled WMMA paragraph (block_size=32), and "Kernel authoring guide",
 *   §4.3 (GFX950 scaled MFMA for MXFP4).  Element value =
 *   e2m1(code) * 2^(e8m0 - 127).
 * - The E2M1 and E8M0 encodings are not printed on the pages; they follow the
 *   OCP Microscaling Formats (MX) v1.0 definitions: E2M1 has 1 sign, 2
 *   exponent (bias 1) and 1 mantissa bit, no Inf/NaN; E8M0 is 2^(e-127) with
 *   0xFF = NaN.  Packing (two codes per byte) is given only as "2
 *   values/byte" ("FlyDSL Kernel Authoring Skill", §10 Troubleshooting, item
 *   10); the reading taken here is: the even k sits in the low nibble.
 * - bf16 output rounding: the pages cast f32 -> bf16 (`.to(fx.BFloat16)`,
 *   §3 "Internal Types") without naming a rounding mode; round-to-nearest-
 *   even from the IEEE 754 definition is the reading taken.
 * - Fused epilogue (orc_gemm_fused): the preshuffle GEMM of "Kernel
 *   authoring guide", §11 "Complete example: Preshuffle GEMM", takes
 *   scale_a, scale_b and bias tensors, fp8 or bf16 inputs, bf16 output and
 *   an epilogue among none / bias / bias_relu / bias_silu / bias_gelu, but
 *   does not spell out their arithmetic.  Reading taken, the plainest one:
 *     y[m,n] = act( acc[m,n] * scale_a[m] * scale_b[n] + bias[n] )
 *   with scale_a one fp32 factor per row of A, scale_b one per row of B
 *   (per column of D), bias one fp32 value per column of D (added only by
 *   the bias_* epilogues), and the activation applied last:
 *   relu(y) = max(y, 0); silu(y) = y / (1 + e^-y); gelu(y) = y * Phi(y)
 *   = y/2 * (1 + erf(y / sqrt 2)), the exact (erf) form of GELU, not the
 *   tanh approximation.
 * - W4A8 (orc_gemm_w4a8): "FlyDSL Kernel Authoring Skill", §10
 *   Troubleshooting, item 10: A is int8, B is packed int4, two values per
 *   byte, unpacked to int8 in the kernel; the integer atoms accumulate in
 *   int32 (§6, the i8 -> i32 and i4 -> i32 WMMA rows, signed operands).
 *   Readings: the even k sits in the low nibble (as for fp4), a nibble is a
 *   4-bit two's complement integer in [-8, 7], and D is the exact integer
 *   sum (int64 here; the library returns int32).
 * - fp8 inputs: the pages' fp8 atoms use Float8E4M3FNUZ on CDNA3 ("FlyDSL
 *   Kernel Authoring Skill", §6).  The E4M3 read here is the OCP 8-bit
 *   floating point format E4M3 (bias 7, no infinities, S.1111.111 = NaN,
 *   largest finite 448), the FP8 format of the GB300 tensor cores.
 *
 * Every function here is pinned by tests/test_oracle_pins.py against values
 * the pages print, closed forms, brute force and independent libraries.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* A rank-2 layout: two top-level modes (row mode, column mode), each with
 * one or two sub-modes.  shape/stride counted in elements. */
typedef struct {
    int32_t depth[2];
    int64_t shape[2][2];
    int64_t stride[2][2];
} orc_layout;

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

/* ---------------------------------------------------------------- layouts */

/* Offset contributed by one top-level mode for scalar coordinate c. */
static int64_t mode_offset(const orc_layout *L, int t, int64_t c)
{
    if (L->depth[t] == 1)
        return c * L->stride[t][0];
    /* nested mode (s0, s1):(d0, d1): split c colexicographically */
    int64_t c0 = c % L->shape[t][0];
    int64_t c1 = c / L->shape[t][0];
    return c0 * L->stride[t][0] + c1 * L->stride[t][1];
}

/* crd2idx: index = sum over modes of coordinate * stride. */
int64_t orc_crd2idx(int64_t row, int64_t col, const orc_layout *L)
{
    return mode_offset(L, 0, row) + mode_offset(L, 1, col);
}

/* idx2crd over the top-level shape: colexicographic, first mode fastest.
 * Writes (row, col).  The shape of mode t is the product of its sub-modes. */
void orc_idx2crd(int64_t idx, const orc_layout *L, int64_t *row, int64_t *col)
{
    int64_t s0 = L->shape[0][0] * (L->depth[0] == 2 ? L->shape[0][1] : 1);
    *row = idx % s0;
    *col = idx / s0;
}

/* Size of top-level mode t. */
int64_t orc_mode_size(const orc_layout *L, int t)
{
    return L->shape[t][0] * (L->depth[t] == 2 ? L->shape[t][1] : 1);
}

/* -------------------------------------------------------------- decoding */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
double orc_decode_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double orc_decode_f32(uint32_t bits)
{
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* OCP MX E2M1: s | e1 e0 | m.  e == 0 is subnormal: (m/2) * 2^(1-bias),
 * bias 1.  Otherwise (1 + m/2) * 2^(e-1). */
double orc_decode_e2m1(uint8_t code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* OCP FP8 E4M3: s | e3 e2 e1 e0 | m2 m1 m0, bias 7.  e == 0 is subnormal:
 * (m/8) * 2^-6.  e == 15 with m == 7 is NaN (no infinities).  Otherwise
 * (1 + m/8) * 2^(e-7). */
double orc_decode_e4m3(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* OCP MX E8M0: 2^(byte - 127); 0xFF encodes NaN. */
double orc_decode_e8m0(uint8_t byte)
{
    if (byte == 0xFF)
        return NAN;
    return ldexp(1.0, (int)byte - 127);
}

/* Round a real value to the nearest bf16 (ties to even), IEEE 754 rules:
 * 8 significant bits, exponent range [-126, 127], subnormal quantum 2^-133,
 * overflow to infinity.  Returns the bf16 bit pattern. */
uint16_t orc_round_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (isinf(ax))
        return sign | 0x7F80;
    if (ax == 0.0)
        return sign;
    int E;
    frexp(ax, &E);                    /* ax in [2^(E-1), 2^E) */
    int qexp = E - 8;                 /* quantum of an 8-bit significand */
    if (qexp < -133)
        qexp = -133;                  /* subnormal range */
    double r = ldexp(ax, -qexp);      /* exact: power-of-two scaling */
    double fl = floor(r);
    double frac = r - fl;
    double n = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))
        n = fl + 1.0;
    double v = ldexp(n, qexp);
    if (v >= ldexp(1.0, 128))
        return sign | 0x7F80;         /* overflow */
    float f = (float)v;               /* exact: v has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* orc_round_bf16 over an array. */
void orc_round_bf16_array(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_round_bf16(x[i]);
}

/* Element (r, c) of a matrix with the given layout and element type. */
static double fetch(const void *X, const orc_layout *L, int dtype,
                    int64_t r, int64_t c)
{
    int64_t i = orc_crd2idx(r, c, L);
    if (dtype == ORC_BF16)
        return orc_decode_bf16(((const uint16_t *)X)[i]);
    if (dtype == ORC_E4M3)
        return orc_decode_e4m3(((const uint8_t *)X)[i]);
    return orc_decode_f32(((const uint32_t *)X)[i]);
}

/* Decode an R x C matrix through its layout into dense row-major fp64. */
int orc_read_matrix(const void *X, const orc_layout *L, int dtype,
                    int64_t R, int64_t C, double *out)
{
    if (!X || !L || !out || R < 0 || C < 0)
        return 1;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            out[r * C + c] = fetch(X, L, dtype, r, c);
    return 0;
}

/* MXFP4 element (r, k) of a packed (R, K/2)-byte matrix with its (R, K/32)
 * e8m0 scales, both row-major. */
static double fetch_mxfp4(const uint8_t *X, const uint8_t *S, int64_t K,
                          int64_t r, int64_t k)
{
    uint8_t byte = X[r * (K / 2) + k / 2];
    uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0x0F);
    uint8_t sc = S[r * (K / 32) + k / 32];
    return orc_decode_e2m1(code) * orc_decode_e8m0(sc);
}

/* ------------------------------------------------------------------ GEMM */

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* The contraction over decoded fp64 operands, a: M x K, b: N x K, both dense
 * row-major.  One fp64 sum per output, k in increasing order. */
static void contract(const double *a, const double *b, int64_t M, int64_t N,
                     int64_t K, double *d)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += a[m * K + k] * b[n * K + k];
            d[m * N + n] = s;
        }
}

/* D (M x N dense row-major fp64) = A·Bᵀ for fp32 / bf16 operands given
 * through layouts over (m,k) and (n,k). */
int orc_gemm(const void *A, const orc_layout *LA, const void *B,
             const orc_layout *LB, int dtype, int64_t M, int64_t N, int64_t K,
             double *D, int nthreads)
{
    if (!A || !B || !LA || !LB || !D || M < 0 || N < 0 || K < 0)
        return 1;
    set_threads(nthreads);
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K + 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(N * K + 1));
    if (!a || !b) {
        free(a);
        free(b);
        return 2;
    }
    orc_read_matrix(A, LA, dtype, M, K, a);
    orc_read_matrix(B, LB, dtype, N, K, b);
    contract(a, b, M, N, K, D);
    free(a);
    free(b);
    return 0;
}

/* Selected entries D[ms[i], ns[i]], each summed directly from the encoded
 * operands (no decode pass) — for spot checks of large problems. */
int orc_gemm_entries(const void *A, const orc_layout *LA, const void *B,
                     const orc_layout *LB, int dtype, int64_t K,
                     const int64_t *ms, const int64_t *ns, int64_t count,
                     double *out, int nthreads)
{
    if (!A || !B || !LA || !LB || !ms || !ns || !out || count < 0)
        return 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += fetch(A, LA, dtype, ms[i], k) * fetch(B, LB, dtype, ns[i], k);
        out[i] = s;
    }
    return 0;
}

/* MXFP4: D (M x N dense row-major fp64) = A·Bᵀ with
 * a(m,k) = e2m1(A code) * 2^(sA[m, k/32] - 127), likewise b(n,k). */
int orc_gemm_mxfp4(const uint8_t *A, const uint8_t *B, const uint8_t *SA,
                   const uint8_t *SB, int64_t M, int64_t N, int64_t K,
                   double *D, int nthreads)
{
    if (!A || !B || !SA || !SB || !D || M < 0 || N < 0 || K < 0 || K % 32)
        return 1;
    set_threads(nthreads);
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K + 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(N * K + 1));
    if (!a || !b) {
        free(a);
        free(b);
        return 2;
    }
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            a[m * K + k] = fetch_mxfp4(A, SA, K, m, k);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            b[n * K + k] = fetch_mxfp4(B, SB, K, n, k);
    contract(a, b, M, N, K, D);
    free(a);
    free(b);
    return 0;
}

int orc_gemm_mxfp4_entries(const uint8_t *A, const uint8_t *B,
                           const uint8_t *SA, const uint8_t *SB, int64_t K,
                           const int64_t *ms, const int64_t *ns, int64_t count,
                           double *out, int nthreads)
{
    if (!A || !B || !SA || !SB || !ms || !ns || !out || count < 0 || K % 32)
        return 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += fetch_mxfp4(A, SA, K, ms[i], k) * fetch_mxfp4(B, SB, K, ns[i], k);
        out[i] = s;
    }
    return 0;
}

/* Decode a packed (R, K/2)-byte MXFP4 matrix with its scales to fp64. */
int orc_read_mxfp4(const uint8_t *X, const uint8_t *S, int64_t R, int64_t K,
                   double *out)
{
    if (!X || !S || !out || K % 32)
        return 1;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            out[r * K + k] = fetch_mxfp4(X, S, K, r, k);
    return 0;
}

/* ------------------------------------------------------- fused epilogue */

enum { ORC_EPI_NONE = 0, ORC_EPI_BIAS = 1, ORC_EPI_BIAS_RELU = 2,
       ORC_EPI_BIAS_SILU = 3, ORC_EPI_BIAS_GELU = 4 };

/* The activation of an epilogue, in fp64 (identity for none / bias). */
double orc_activation(double y, int epi)
{
    switch (epi) {
    case ORC_EPI_BIAS_RELU:
        return y > 0.0 ? y : 0.0;
    case ORC_EPI_BIAS_SILU:
        return y / (1.0 + exp(-y));
    case ORC_EPI_BIAS_GELU:
        return 0.5 * y * (1.0 + erf(y / sqrt(2.0)));
    default:
        return y;
    }
}

/* act(acc * sa[m] * sb[n] + bias[n]) for one output; sa / sb may be NULL
 * (factor 1); bias is read only by the bias_* epilogues. */
static double epilogue(double acc, int64_t m, int64_t n, const float *sa,
                       const float *sb, const float *bias, int epi)
{
    double y = acc;
    if (sa)
        y *= (double)sa[m];
    if (sb)
        y *= (double)sb[n];
    if (epi >= ORC_EPI_BIAS)
        y += (double)bias[n];
    return orc_activation(y, epi);
}

/* Fused GEMM: A (M,K) and B (N,K) dense row-major in `dtype` (bf16 or
 * E4M3); D (M x N dense row-major fp64) before the bf16 output rounding. */
int orc_gemm_fused(const void *A, const void *B, int dtype, int64_t M,
                   int64_t N, int64_t K, const float *sa, const float *sb,
                   const float *bias, int epi, double *D, int nthreads)
{
    if (!A || !B || !D || M < 0 || N < 0 || K < 0 || epi < 0 || epi > 4 ||
        (epi >= ORC_EPI_BIAS && !bias) || (dtype != ORC_BF16 && dtype != ORC_E4M3))
        return 1;
    orc_layout la, lb;
    memset(&la, 0, sizeof la);
    memset(&lb, 0, sizeof lb);
    la.depth[0] = la.depth[1] = lb.depth[0] = lb.depth[1] = 1;
    la.shape[0][0] = M;
    la.shape[1][0] = K;
    la.stride[0][0] = K;
    la.stride[1][0] = 1;
    lb.shape[0][0] = N;
    lb.shape[1][0] = K;
    lb.stride[0][0] = K;
    lb.stride[1][0] = 1;
    int rc = orc_gemm(A, &la, B, &lb, dtype, M, N, K, D, nthreads);
    if (rc)
        return rc;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            D[m * N + n] = epilogue(D[m * N + n], m, n, sa, sb, bias, epi);
    return 0;
}

/* Selected outputs of orc_gemm_fused, each summed directly. */
int orc_gemm_fused_entries(const void *A, const void *B, int dtype, int64_t K,
                           const float *sa, const float *sb, const float *bias,
                           int epi, const int64_t *ms, const int64_t *ns,
                           int64_t count, double *out, int nthreads)
{
    if (!A || !B || !ms || !ns || !out || count < 0 || epi < 0 || epi > 4 ||
        (epi >= ORC_EPI_BIAS && !bias) || (dtype != ORC_BF16 && dtype != ORC_E4M3))
        return 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        const int64_t m = ms[i], n = ns[i];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = dtype == ORC_BF16 ? orc_decode_bf16(((const uint16_t *)A)[m * K + k])
                                         : orc_decode_e4m3(((const uint8_t *)A)[m * K + k]);
            double b = dtype == ORC_BF16 ? orc_decode_bf16(((const uint16_t *)B)[n * K + k])
                                         : orc_decode_e4m3(((const uint8_t *)B)[n * K + k]);
            s += a * b;
        }
        out[i] = epilogue(s, m, n, sa, sb, bias, epi);
    }
    return 0;
}

/* ------------------------------------------------------------------ W4A8 */

/* Signed 4-bit two's complement: 0..7 -> 0..7, 8..15 -> -8..-1. */
int orc_decode_int4(uint8_t nibble)
{
    nibble &= 0x0F;
    return nibble >= 8 ? (int)nibble - 16 : (int)nibble;
}

/* Element (n, k) of a packed (N, K/2)-byte int4 matrix, row-major. */
static int fetch_int4(const uint8_t *B, int64_t K, int64_t n, int64_t k)
{
    uint8_t byte = B[n * (K / 2) + k / 2];
    return orc_decode_int4((k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0x0F));
}

/* D (M x N, int64) = sum_k a(m,k) * b(n,k), exactly: A (M, K) int8
 * row-major, B (N, K/2) packed int4 row-major. */
int orc_gemm_w4a8(const int8_t *A, const uint8_t *B, int64_t M, int64_t N,
                  int64_t K, int64_t *D, int nthreads)
{
    if (!A || !B || !D || M < 0 || N < 0 || K < 0 || K % 2)
        return 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k)
                s += (int64_t)A[m * K + k] * fetch_int4(B, K, n, k);
            D[m * N + n] = s;
        }
    return 0;
}

/* Selected outputs of orc_gemm_w4a8. */
int orc_gemm_w4a8_entries(const int8_t *A, const uint8_t *B, int64_t K,
                          const int64_t *ms, const int64_t *ns, int64_t count,
                          int64_t *out, int nthreads)
{
    if (!A || !B || !ms || !ns || !out || count < 0 || K % 2)
        return 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        int64_t s = 0;
        for (int64_t k = 0; k < K; ++k)
            s += (int64_t)A[ms[i] * K + k] * fetch_int4(B, K, ns[i], k);
        out[i] = s;
    }
    return 0;
}
