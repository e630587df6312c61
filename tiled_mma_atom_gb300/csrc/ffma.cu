// ffma.cu — CUDA-core fp32 FMA kernels.
//
// 1. ffma_gemm: D = A·Bᵀ for any (Shape, Stride) layouts of A, B and D, fp32
//    or bf16 elements, fp32 accumulation.  Every global address is the
//    layout's crd2idx of the logical coordinate ("FlyDSL Kernel Authoring
//    Skill", §2 "Coordinate Mapping": index = sum of coordinate x stride; a
//    nested mode's scalar coordinate is split first-sub-mode-fastest).  The
//    page's "Naive GEMM Template" (§8) computes one output per thread with a
//    K loop of scalar loads; here a CTA stages 16-deep K slices of a 64x64 (or
//    32x32) output tile in shared memory and each thread accumulates a
//    register tile, summing k in increasing order.
//
// 2. skinny_ffma: M <= 16 decode-shaped GEMM with K-major bf16 operands.  A
//    warp streams four rows of B with 128-bit loads, lanes splitting K, and
//    reduces the per-lane partial sums with warp shuffles (the warp
//    reduction of §7 "Reduction Patterns", on 32-lane warps).
#include <cuda_bf16.h>

#include "internal.h"

namespace tmg {
namespace {

__device__ __forceinline__ int64_t mode_off(const DevLayout &L, int t, int64_t c)
{
    if (L.depth[t] == 1)
        return c * L.stride[t][0];
    const int64_t s0 = L.shape[t][0];
    return (c % s0) * L.stride[t][0] + (c / s0) * L.stride[t][1];
}

__device__ __forceinline__ int64_t crd2idx(const DevLayout &L, int64_t r, int64_t c)
{
    return mode_off(L, 0, r) + mode_off(L, 1, c);
}

template <typename T>
__device__ __forceinline__ float ld_elt(const T *p, int64_t i);
template <>
__device__ __forceinline__ float ld_elt<float>(const float *p, int64_t i)
{
    return __ldg(p + i);
}
template <>
__device__ __forceinline__ float ld_elt<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i)
{
    return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st_elt(T *p, int64_t i, float v);
template <>
__device__ __forceinline__ void st_elt<float>(float *p, int64_t i, float v)
{
    p[i] = v;
}
template <>
__device__ __forceinline__ void st_elt<__nv_bfloat16>(__nv_bfloat16 *p, int64_t i, float v)
{
    p[i] = __float2bfloat16_rn(v);
}

constexpr int kFfmaThreads = 256;
constexpr int kFfmaBK = 16;

// Thread (tx, ty) of a 16x16 grid owns rows ty + 16 i and columns tx + 16 j
// of the CTA tile, i < BM/16, j < BN/16.
template <typename T, int BM, int BN>
__global__ void __launch_bounds__(kFfmaThreads)
    ffma_gemm_kernel(const T *__restrict__ A, const T *__restrict__ B, T *__restrict__ D,
                     DevLayout la, DevLayout lb, DevLayout ld, int64_t M, int64_t N, int64_t K)
{
    constexpr int TM = BM / 16, TN = BN / 16;
    __shared__ float As[kFfmaBK][BM + 1];
    __shared__ float Bs[kFfmaBK][BN + 1];

    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j)
            acc[i][j] = 0.f;

    for (int64_t k0 = 0; k0 < K; k0 += kFfmaBK) {
        // k fastest across threads: row-major operands read 64-byte runs
        for (int e = tid; e < BM * kFfmaBK; e += kFfmaThreads) {
            const int kk = e % kFfmaBK, mm = e / kFfmaBK;
            const int64_t m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < M && k < K) ? ld_elt(A, crd2idx(la, m, k)) : 0.f;
        }
        for (int e = tid; e < BN * kFfmaBK; e += kFfmaThreads) {
            const int kk = e % kFfmaBK, nn = e / kFfmaBK;
            const int64_t n = n0 + nn, k = k0 + kk;
            Bs[kk][nn] = (n < N && k < K) ? ld_elt(B, crd2idx(lb, n, k)) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kFfmaBK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i)
                a[i] = As[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < TN; ++j)
                b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j)
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t m = m0 + ty + 16 * i;
        if (m >= M)
            continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int64_t n = n0 + tx + 16 * j;
            if (n < N)
                st_elt(D, crd2idx(ld, m, n), acc[i][j]);
        }
    }
}

template <typename T>
__global__ void zero_fill_kernel(T *D, DevLayout ld, int64_t M, int64_t N)
{
    const int64_t total = M * N;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = e / N, n = e % N;
        st_elt(D, crd2idx(ld, m, n), 0.f);
    }
}

// --------------------------------------------------------------- skinny

constexpr int kSkR = 4;          // rows of B per warp task
constexpr int kSkMaxM = 16;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Warp task t covers B rows [4t, 4t+4).  Lane l owns k in {8l + 256 i}.
__global__ void __launch_bounds__(256)
    skinny_ffma_kernel(const __nv_bfloat16 *__restrict__ A, const __nv_bfloat16 *__restrict__ B,
                       __nv_bfloat16 *__restrict__ D, int M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldd)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    const int64_t tasks = (N + kSkR - 1) / kSkR;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
         t < tasks; t += warps_total) {
        const int64_t nbase = t * kSkR;
        float acc[kSkR][kSkMaxM];
#pragma unroll
        for (int r = 0; r < kSkR; ++r)
#pragma unroll
            for (int m = 0; m < kSkMaxM; ++m)
                acc[r][m] = 0.f;

        for (int64_t k = 8 * lane; k < K; k += 256) {
            float b[kSkR][8];
#pragma unroll
            for (int r = 0; r < kSkR; ++r) {
                const int64_t n = nbase + r;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (n < N)
                    v = __ldcs(reinterpret_cast<const uint4 *>(B + n * ldb + k));
                bf16x8_to_f32(v, b[r]);
            }
#pragma unroll
            for (int m = 0; m < kSkMaxM; ++m) {
                if (m < M) {
                    float a[8];
                    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(A + m * lda + k)), a);
#pragma unroll
                    for (int r = 0; r < kSkR; ++r)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            acc[r][m] = fmaf(a[i], b[r][i], acc[r][m]);
                }
            }
        }
        // butterfly sum over the 32 lanes
#pragma unroll
        for (int r = 0; r < kSkR; ++r)
#pragma unroll
            for (int m = 0; m < kSkMaxM; ++m) {
                float v = acc[r][m];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
                acc[r][m] = v;
            }
        // lane (r * 16 + m) writes output (m, nbase + r) — 64 lanes' worth
        // of values, so two passes of the warp
#pragma unroll
        for (int r = 0; r < kSkR; ++r)
#pragma unroll
            for (int m = 0; m < kSkMaxM; ++m)
                if (lane == ((r * kSkMaxM + m) & 31) && m < M && nbase + r < N)
                    D[m * ldd + nbase + r] = __float2bfloat16_rn(acc[r][m]);
    }
}

}  // namespace

cudaError_t launch_ffma(const FfmaArgs &a, int dtype, int num_sms, const ErrCtx &err,
                        cudaStream_t s)
{
    (void)err;
    // small problems: 32x32 tiles for more CTAs; else 64x64
    const bool small = (a.M * a.N) <= static_cast<int64_t>(num_sms) * 64 * 64;
    const int bm = small ? 32 : 64;
    dim3 grid(static_cast<unsigned>((a.N + bm - 1) / bm), static_cast<unsigned>((a.M + bm - 1) / bm));
    if (grid.y > 65535u)
        return cudaErrorInvalidConfiguration;
    note_launch();
    if (dtype == 0) {
        const float *A = static_cast<const float *>(a.A), *B = static_cast<const float *>(a.B);
        float *D = static_cast<float *>(a.D);
        if (small)
            ffma_gemm_kernel<float, 32, 32><<<grid, kFfmaThreads, 0, s>>>(A, B, D, a.la, a.lb, a.ld, a.M, a.N, a.K);
        else
            ffma_gemm_kernel<float, 64, 64><<<grid, kFfmaThreads, 0, s>>>(A, B, D, a.la, a.lb, a.ld, a.M, a.N, a.K);
    } else {
        const __nv_bfloat16 *A = static_cast<const __nv_bfloat16 *>(a.A);
        const __nv_bfloat16 *B = static_cast<const __nv_bfloat16 *>(a.B);
        __nv_bfloat16 *D = static_cast<__nv_bfloat16 *>(a.D);
        if (small)
            ffma_gemm_kernel<__nv_bfloat16, 32, 32><<<grid, kFfmaThreads, 0, s>>>(A, B, D, a.la, a.lb, a.ld, a.M, a.N, a.K);
        else
            ffma_gemm_kernel<__nv_bfloat16, 64, 64><<<grid, kFfmaThreads, 0, s>>>(A, B, D, a.la, a.lb, a.ld, a.M, a.N, a.K);
    }
    return cudaGetLastError();
}

cudaError_t launch_zero_fill(void *D, const DevLayout &ld, int64_t M, int64_t N, int dtype,
                             cudaStream_t s)
{
    const int64_t total = M * N;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > 4096)
        blocks = 4096;
    if (blocks < 1)
        blocks = 1;
    note_launch();
    if (dtype == 0)
        zero_fill_kernel<float><<<blocks, 256, 0, s>>>(static_cast<float *>(D), ld, M, N);
    else
        zero_fill_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<__nv_bfloat16 *>(D), ld, M, N);
    return cudaGetLastError();
}

cudaError_t launch_skinny_ffma(const SkinnyFfmaArgs &a, int num_sms, cudaStream_t s)
{
    const int64_t tasks = (a.N + kSkR - 1) / kSkR;
    int64_t blocks = (tasks + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap)
        blocks = cap;
    note_launch();
    skinny_ffma_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(a.A), static_cast<const __nv_bfloat16 *>(a.B),
        static_cast<__nv_bfloat16 *>(a.D), static_cast<int>(a.M), a.N, a.K, a.lda, a.ldb, a.ldd);
    return cudaGetLastError();
}

}  // namespace tmg
