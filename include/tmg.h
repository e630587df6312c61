/*
 * tmg.h — C ABI of the GB300 tiled GEMM library (libtmg.so).
 *
 * The library computes D = A·Bᵀ with fp32 accumulation on one NVIDIA GB300
 * (sm_103a) GPU.  All compute runs in the library's own CUDA kernels; there
 * is no CPU fallback: a call either launches GPU work or returns an error.
 *
 * Operation, as the FlyDSL pages state it:
 *   - Operand convention A = (M,K), B = (N,K), C/D = (M,N): "add-target-atom-op"
 *     (skillsmp.com), §1.4 "ThrVal layouts describe the per-thread register
 *     footprint" and §1.5.3 "Reference coordinate system is column-major".
 *   - Layouts are (Shape, Stride) pairs; element (i,j) lives at
 *     crd2idx((i,j)) = i*stride_0 + j*stride_1: "FlyDSL Kernel Authoring
 *     Skill", §2 "Layout System", "Core Types" and "Coordinate Mapping".
 *     A top-level mode may be nested one level, e.g. (9,(4,8)) ("Construction"
 *     in the same section); a scalar coordinate of a nested mode is split
 *     colexicographically (first sub-mode fastest), the order idx2crd uses
 *     in the worked example of "Coordinate Mapping".
 *   - fp32 accumulation: the f32-accumulating MFMA atoms of §6 "MFMA
 *     Integration" (e.g. 16x16x4 f32 and 16x16x16 f16/bf16 -> f32).
 *   - bf16 output is the f32 accumulator rounded to nearest even (the pages
 *     write `.to(fx.BFloat16)`, §3 "Internal Types", without a mode).
 *   - MXFP4: e2m1 values with one e8m0 scale per 32 consecutive K elements:
 *     §6, "gfx1250 WMMA (wave32)", MX-scaled WMMA (block_size=32), and
 *     "Kernel authoring guide" (rocm.github.io), §4.3 GFX950 scaled MFMA.
 *   - Calls are asynchronous on a caller-supplied stream: "Kernel authoring
 *     guide", §2.4 `fx.Stream`.
 *
 * Ownership: the caller owns every buffer passed in (device memory, e.g.
 * torch tensors).  The library never frees or retains them beyond the
 * call.  The library owns only: a device error word (static device memory)
 * and per-(device, stream) scratch — split-K partials for the skinny path,
 * stream-K partial tiles for the CTA-pair kernels, relaid scales for the
 * MXFP4 path, packed operands of the general-layout path — grown on demand
 * and released by tmg_shutdown().
 *
 * Errors: nothing is allowed to fault.  Bad arguments return
 * TMG_ERR_INVALID_ARG, valid but unhandled requests TMG_ERR_UNSUPPORTED,
 * CUDA launch/runtime failures TMG_ERR_CUDA.  Every wait inside a kernel is
 * bounded; a wait that runs out sets the device error word and the kernel
 * returns early — tmg_check() then reports TMG_ERR_TIMEOUT.
 * tmg_last_error() gives a message for the calling thread's last failure.
 *
 * Debug aids.  TMG_LOG=1 in the environment makes every GEMM call print the
 * kernel family, tile and schedule it chose (one line on stderr).  The
 * library also builds as libtmg_debug.so (same ABI; build.py
 * --debug-bounds): there every store of D and every access to split-K
 * scratch is checked against its buffer, an out-of-range offset skips the
 * access and sets the device error word, and tmg_check() then reports
 * TMG_ERR_BOUNDS.
 */
#ifndef TMG_H
#define TMG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TMG_OK = 0,
    TMG_ERR_INVALID_ARG = 1,
    TMG_ERR_UNSUPPORTED = 2,
    TMG_ERR_CUDA = 3,
    TMG_ERR_TIMEOUT = 4,
    TMG_ERR_BOUNDS = 5      /* debug build only: a kernel caught an out-of-range offset */
} tmg_status;

/* Element type.  tmg_gemm: the type of A, B and D (identical), F32 or BF16.
 * tmg_gemm_fused: the type of A and B, BF16 or E4M3 (D is bf16).
 * Accumulation is always fp32.  E4M3 is the OCP 8-bit floating point format
 * (sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities;
 * S.1111.111 is NaN; largest finite value 448). */
typedef enum { TMG_F32 = 0, TMG_BF16 = 1, TMG_E4M3 = 2 } tmg_dtype;

/* Epilogue of tmg_gemm_fused, applied to each fp32 result before the bf16
 * rounding: y = acc * scale_a[m] * scale_b[n], then for the BIAS variants
 * y += bias[n], then the activation:
 *   RELU: max(y, 0);  SILU: y / (1 + exp(-y));
 *   GELU: y/2 * (1 + erf(y / sqrt(2)))  (the erf form, not the tanh one). */
typedef enum {
    TMG_EPI_NONE = 0,
    TMG_EPI_BIAS = 1,
    TMG_EPI_BIAS_RELU = 2,
    TMG_EPI_BIAS_SILU = 3,
    TMG_EPI_BIAS_GELU = 4
} tmg_epilogue;

/* Which kernel family runs a gemm.  AUTO picks by dtype, layout and shape:
 *   FFMA   — CUDA-core fp32 FMA, any layout (the fp32 path, and the general
 *            layout path for bf16);
 *   TC     — persistent tcgen05 tensor-core GEMM, bf16, K-major operands;
 *   SKINNY — tensor-core swap-AB split-K GEMM for M <= 64, bf16, K-major;
 *   SKINNY_FFMA — CUDA-core split-K dot products for M <= 16, bf16, K-major;
 *   TC_SINGLE / TC_PAIR — TC restricted to one-CTA 128-row tiles or to
 *            CTA-pair (cta_group::2) 256-row tiles; TC picks between them;
 *   PACKED_TC — bf16 in any layout on the tensor cores.  Flat MN-major
 *            operands (A as (M,K):(1,lda), B as (N,K):(1,ldb), i.e. B stored
 *            K x N row-major as in C = A*B; 16-byte aligned, ld a multiple
 *            of 8) are read in place by the CTA-pair kernel when D is
 *            row-major, M >= 256 and the pair tiles fill every pair once;
 *            otherwise operands the TMA cannot read in place (MN-major,
 *            nested, strided, broadcast) are first gathered through their
 *            layouts into K-major workspace copies, and a D that is neither
 *            row- nor column-major is computed into a dense workspace and
 *            scattered back.  AUTO takes it for bf16 problems with
 *            M*N*K >= 2^27 that TC cannot read in place (smaller ones go to
 *            FFMA).
 * Forcing a family that cannot take the arguments returns UNSUPPORTED. */
typedef enum {
    TMG_PATH_AUTO = 0,
    TMG_PATH_FFMA = 1,
    TMG_PATH_TC = 2,
    TMG_PATH_SKINNY = 3,
    TMG_PATH_SKINNY_FFMA = 4,
    TMG_PATH_TC_SINGLE = 5,
    TMG_PATH_TC_PAIR = 6,
    TMG_PATH_PACKED_TC = 7
} tmg_path;

/* A rank-2 layout over logical coordinates (row, col).  Mode t (0 = rows,
 * 1 = columns) has depth[t] sub-modes (1 or 2) with shapes shape[t][0..] and
 * strides stride[t][0..], counted in elements.  Unused entries are ignored.
 * The product of the sub-shapes of mode t must equal the logical extent.
 * Example: a row-major M x K matrix with leading dimension ld is
 * {depth={1,1}, shape={{M,1},{K,1}}, stride={{ld,0},{1,0}}}. */
typedef struct {
    int32_t depth[2];
    int64_t shape[2][2];
    int64_t stride[2][2];
} tmg_layout;

/* D[m,n] = sum_k A(m,k) * B(n,k), fp32 accumulation.
 *   A, B, D  device pointers to the element type `dtype`.
 *   M, N, K  logical extents, each >= 0.  M == 0 or N == 0 is a no-op;
 *            K == 0 writes zeros to D.
 *   layoutA  over (m,k); NULL means row-major (M,K):(K,1).
 *   layoutB  over (n,k); NULL means row-major (N,K):(K,1).
 *   layoutD  over (m,n); NULL means row-major (M,N):(N,1).  D's layout must
 *            map distinct (m,n) to distinct elements (strides > 0).
 *   stream   a cudaStream_t (NULL = the legacy default stream).
 * Asynchronous: returns after the launch.  Input strides may be 0
 * (broadcast).  Offsets must fit in int64. */
tmg_status tmg_gemm(const void *A, const void *B, void *D, int64_t M, int64_t N,
                    int64_t K, tmg_dtype dtype, const tmg_layout *layoutA,
                    const tmg_layout *layoutB, const tmg_layout *layoutD,
                    void *stream);

/* tmg_gemm with an explicit kernel family (see tmg_path). */
tmg_status tmg_gemm_ex(const void *A, const void *B, void *D, int64_t M,
                       int64_t N, int64_t K, tmg_dtype dtype,
                       const tmg_layout *layoutA, const tmg_layout *layoutB,
                       const tmg_layout *layoutD, tmg_path path, void *stream);

/* tmg_gemm from host memory: the same D = A·Bᵀ with row-major operands in
 * HOST buffers (pinned memory recommended; pageable memory works, slower):
 *   A  host, (M, K) row-major of `dtype` (TMG_F32 or TMG_BF16)
 *   B  host, (N, K) row-major;  D  host, (M, N) row-major, written.
 * The library copies B to device workspace, then pipelines row chunks of A
 * and D: the upload of chunk i+1, the GEMM of chunk i (on `stream`, through
 * the tmg_gemm dispatch) and the download of chunk i-1 overlap on two
 * library-owned copy streams.  Asynchronous: on return the work is queued
 * and `stream` waits for the last download; synchronise `stream` before
 * reading D or reusing A and B.  Device pointers are rejected
 * (INVALID_ARG).  Workspace (M·K + N·K + M·N elements), copy streams and
 * events are per (device, stream), grown on demand, freed by tmg_shutdown().
 * The FlyDSL pages have no host-memory entry; this is the library's
 * end-to-end call. */
tmg_status tmg_gemm_host(const void *A, const void *B, void *D, int64_t M,
                         int64_t N, int64_t K, tmg_dtype dtype, void *stream);

/* Fused GEMM: D[m,n] = bf16_rne( act( (sum_k a(m,k) * b(n,k)) * scale_a[m]
 * * scale_b[n] + bias[n] ) ), fp32 accumulation.  The options mirror the
 * preshuffle GEMM of "Kernel authoring guide" (rocm.github.io), §11
 * "Complete example: Preshuffle GEMM": fp8 or bf16 inputs, bf16 output,
 * optional scale_a / scale_b / bias tensors and the epilogues none, bias,
 * bias_relu, bias_silu, bias_gelu.  The pages do not spell out how these
 * combine; the reading taken is the formula above (scale_a by row of A,
 * scale_b by row of B, bias by column of D, activation last).
 *   A         device, (M, K) row-major, K contiguous, of type in_dtype.
 *   B         device, (N, K) row-major, K contiguous, of type in_dtype.
 *   D         device, bf16 (M, N) row-major.
 *   in_dtype  TMG_BF16 or TMG_E4M3 (TMG_F32: UNSUPPORTED).
 *   scale_a   device fp32 [M] or NULL (all ones).
 *   scale_b   device fp32 [N] or NULL (all ones).
 *   bias      device fp32 [N]; required (else INVALID_ARG) by the BIAS
 *             epilogues, ignored by TMG_EPI_NONE.
 * K == 0 gives D = act(bias) (zeros for TMG_EPI_NONE).  Tensor-core kernel
 * (CTA pairs, kind::f16 or kind::f8f6f4): A, B 16-byte aligned and K times
 * the element size a multiple of 16 bytes (else UNSUPPORTED).  The caller
 * owns all buffers; the library reuses its per-(device, stream) stream-K
 * scratch. */
tmg_status tmg_gemm_fused(const void *A, const void *B, void *D, int64_t M,
                          int64_t N, int64_t K, tmg_dtype in_dtype,
                          const float *scale_a, const float *scale_b,
                          const float *bias, tmg_epilogue epilogue,
                          void *stream);

/* W4A8 GEMM: D[m,n] = sum_k a(m,k) * b(n,k), exact, as int32.
 *   A  device, (M, K) int8 row-major.
 *   B  device, (N, K/2) bytes row-major: packed signed int4 (two's
 *      complement, -8..7), the even k in the low nibble (bits 0-3).
 *   D  device, int32 (M, N) row-major.
 * "FlyDSL Kernel Authoring Skill", §10 Troubleshooting, item 10 (int8 A,
 * packed int4 B unpacked in the kernel) and §6 (i8 / i4 atoms accumulating
 * in i32).  K must be even (else INVALID_ARG); K == 0 writes zeros; results
 * wrap like int32 arithmetic only if |D| >= 2^31 (K > 2^21 with extreme
 * values).  GB300 has no integer tensor-core MMA, so exact integer sums are
 * formed on floating-point tensor cores:
 *   decode shapes (M <= 64, K a multiple of 32, K <= 32768): the weights
 *     stay 4-bit until the kernel, which turns them into offset-binary E4M3
 *     codes (u = b + 8; code u is exactly u * 2^-9) in tensor memory, splits
 *     a = 16 hi + lo (both exact in E4M3) and multiplies on the fp8 tensor
 *     cores; every fp32 column sum is an integer multiple of 2^-9 below 2^22
 *     in magnitude, and the epilogue subtracts 8 * sum_k a(m,k); CTAs that
 *     share an output tile add their int32 shares into D.  Workspace:
 *     2 * round_up(M, 16) * K + 4 * round_up(M, 16) bytes per (device,
 *     stream);
 *   otherwise: both operands are unpacked to bf16 (exact) into workspace
 *     ((M + N) x K bf16), multiplied on the bf16 tensor cores in K segments
 *     of at most 8192 — where every fp32 partial sum is an integer of
 *     magnitude at most 2^23, hence exact — and each segment is stored or
 *     added into D as int32. */
tmg_status tmg_gemm_w4a8(const void *A, const void *B, void *D, int64_t M,
                         int64_t N, int64_t K, void *stream);

/* Pre-shuffled W4A8 weights ("FlyDSL Kernel Authoring Skill", §6 GEMM
 * Pattern (Preshuffle): B is rearranged once, offline, so that each tile the
 * kernel reads is contiguous).  The image is a sequence of 16 KB blocks, one
 * per (t, kb) = (128 weight rows, 256 k), block t * ceil(K / 256) + kb; in a
 * block, row r (weight row 128 t + r) takes bytes r * 128 .. r * 128 + 127,
 * and its 16-byte chunk c (k = 256 kb + 32 c .. + 31, packed as in B) sits
 * at chunk slot c XOR (r mod 8).  Rows past N and k past K are zero.
 *
 * tmg_w4a8_preshuffled_bytes: size of the image, 0 unless N > 0, K > 0 and
 *   K is a multiple of 32.  Host only.
 * tmg_w4a8_preshuffle: B (N, K/2) device, row-major packed int4 -> Bs
 *   (device, tmg_w4a8_preshuffled_bytes(N, K) bytes, caller-owned).  Both
 *   16-byte aligned (else INVALID_ARG); K a multiple of 32 (else
 *   INVALID_ARG); N == 0 or K == 0 does nothing.  Asynchronous on `stream`.
 * tmg_gemm_w4a8_preshuffled: tmg_gemm_w4a8 with the pre-shuffled image Bs
 *   in place of B, same results; K a multiple of 32 and Bs 16-byte aligned
 *   (else INVALID_ARG).  The decode kernel then reads each CTA's share of the
 *   weights as one contiguous stream. */
size_t tmg_w4a8_preshuffled_bytes(int64_t N, int64_t K);
tmg_status tmg_w4a8_preshuffle(const void *B, void *Bs, int64_t N, int64_t K,
                               void *stream);
tmg_status tmg_gemm_w4a8_preshuffled(const void *A, const void *Bs, void *D,
                                     int64_t M, int64_t N, int64_t K,
                                     void *stream);

/* MXFP4 GEMM: D[m,n] = sum_k a(m,k) * b(n,k) with
 *   a(m,k) = e2m1(code of A at (m,k)) * 2^(scaleA[m, k/32] - 127), same for b.
 *   A       device, (M, K/2) bytes row-major: two e2m1 codes per byte, the
 *           even k in the low nibble (bits 0-3), the odd k in bits 4-7.
 *   B       device, (N, K/2) bytes, same packing.
 *   scaleA  device, (M, K/32) e8m0 bytes row-major; scaleB (N, K/32).
 *           Byte 0xFF (NaN) propagates NaN.
 *   D       device, bf16 (M, N) row-major.
 * K must be a positive multiple of 32 (else INVALID_ARG); the tensor-core
 * kernel additionally needs K % 256 == 0 and 16-byte aligned rows
 * (else UNSUPPORTED).  E2M1/E8M0 follow the OCP MX v1.0 definitions. */
tmg_status tmg_gemm_mxfp4(const void *A, const void *B, const void *scaleA,
                          const void *scaleB, void *D, int64_t M, int64_t N,
                          int64_t K, void *stream);

/* Skinny bf16 GEMM that allocates nothing.  The FlyDSL pages have no
 * counterpart: this is a library-level variant for callers that may not
 * allocate device memory at call time — e.g. a latency-critical loop that
 * must not call cudaMalloc/cudaFree after start-up (both can synchronise the
 * device), or a plug-in whose host owns all device memory through its own
 * pool and passes in only the operands.
 *
 * Computes the same D = A·Bᵀ as tmg_gemm on the skinny tensor-core path:
 *   A  device, bf16 (M, K) row-major, row stride lda (elements, >= K)
 *   B  device, bf16 (N, K) row-major, row stride ldb (>= K)
 *   D  device, bf16 (M, N) row-major, row stride ldd (>= N)
 * Limits: M <= 64 and N <= 524288 (else TMG_ERR_INVALID_ARG); A and B rows
 * 16-byte aligned (else TMG_ERR_UNSUPPORTED).
 *
 * Its split-K partial sums and tile counters live in one 8 MiB array in the
 * library's static device memory, which every GPU that loads the library
 * holds until the process exits.  No call allocates or frees memory.  The
 * array holds partial sums for every SM up to M = 48; for M from 49 to 64 it
 * holds them for 127 CTAs, so those calls run on at most 127 of the SMs and
 * split K differently from the allocating call: equal results within
 * rounding, not bit for bit (for M <= 48 the two are bit-identical).  The
 * first call on a device looks up that array's device address (once per
 * device, with the device current) and keeps it for the life of the
 * process: make that first call before any stream capture, and do not use
 * the library on a device after cudaDeviceReset.  Every call shares the one
 * array and it keeps the last call's
 * contents: each call clears the counters it uses with an asynchronous
 * memset on `stream` before its kernel.  Calls whose GPU work overlaps (on
 * different streams, or from different threads) race on the array and give
 * wrong results: serialise them. */
tmg_status tmg_gemm_skinny_noalloc(const void *A, const void *B, void *D,
                                   int64_t M, int64_t N, int64_t K,
                                   int64_t lda, int64_t ldb, int64_t ldd,
                                   void *stream);

/* Synchronise `stream`, then report: TMG_ERR_CUDA for a sticky or pending
 * CUDA error, TMG_ERR_TIMEOUT if a kernel's bounded wait ran out since the
 * last check (the device error word is cleared and the skinny-path scratch
 * counters are reset), else TMG_OK. */
tmg_status tmg_check(void *stream);

/* Message for the calling thread's last non-OK status ("" if none).  The
 * pointer stays valid until the thread's next library call. */
const char *tmg_last_error(void);

/* Budget of every bounded wait inside the kernels, in nanoseconds
 * (default 2 s).  Applies to launches made after the call. */
void tmg_set_wait_budget_ns(uint64_t ns);

/* Launch one tiny kernel that waits on a barrier nothing will ever signal,
 * with the given budget; it must give up and set the device error word, so
 * that the next tmg_check() returns TMG_ERR_TIMEOUT.  Exercises the bounded
 * wait of every kernel without any GPU fault or hang. */
tmg_status tmg_debug_wait_timeout(uint64_t budget_ns, void *stream);

/* Debug build only (libtmg_debug.so): launch one tiny kernel whose bounds
 * check sees an offset one past the end of a buffer — it accesses nothing —
 * so that the next tmg_check() returns TMG_ERR_BOUNDS.  Exercises the
 * reporting of the bounds checks without any out-of-range access.  The
 * normal build returns TMG_ERR_UNSUPPORTED. */
tmg_status tmg_debug_bounds_probe(void *stream);

/* 1 in the debug build (bounds-checked kernels), else 0. */
int tmg_debug_build(void);

/* Number of kernels the library has launched in this process. */
uint64_t tmg_launch_count(void);

/* Library version, major*10000 + minor*100 + patch. */
int tmg_version(void);

/* Free library-owned device scratch and host caches.  Calls already queued
 * must have finished.  The library stays usable afterwards. */
void tmg_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* TMG_H */
