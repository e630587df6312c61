// ffma.cu — CUDA-core fp32 FMA kernels.
//
// 1. ffma_gemm: D = A·Bᵀ for any (Shape, Stride) layouts of A, B and D, fp32
//    or bf16 elements, fp32 accumulation.  Every global address is the
//    layout's crd2idx of the logical coordinate ("FlyDSL Kernel Authoring
//    Skill", §2 "Coordinate Mapping": index = sum of coordinate x stride; a
//    nested mode's scalar coordinate is split first-sub-mode-fastest).  The
//    page's "Naive GEMM Template" (§8) computes one output per thread with a
//    K loop of scalar loads; here a CTA stages 32-deep K slices of a 64x64 (or
//    32x32) output tile in shared memory, prefetching the next slice into
//    registers (the prologue / loop-carried prefetch of §3 "Runtime Loops with
//    Loop-Carried Values"), and each thread accumulates a register tile,
//    summing k in increasing order.  Row-major operands with 16-byte rows
//    take ffma_dense_kernel: the same tiles and k order with 16-byte vector
//    loads at plain row-major addresses.
//
// 2. skinny_ffma: M <= 16 decode-shaped GEMM with K-major bf16 operands.  A
//    warp streams four rows of B with 128-bit loads, lanes splitting K, and
//    reduces the per-lane partial sums with warp shuffles (the warp
//    reduction of §7 "Reduction Patterns", on 32-lane warps).
#include <cuda_bf16.h>

#include "layout.cuh"

namespace tmg {
namespace {

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

// Thread (tx, ty) of a 16x16 grid owns rows ty + 16 i and columns tx + 16 j
// of the CTA tile, i < BM/16, j < BN/16.  Software-pipelined: while the
// threads multiply the K slice in shared memory, the next slice's elements
// are already in flight into registers; two shared buffers alternate, so one
// barrier per slice suffices.  Each output still sums k in increasing order.
template <typename T, int BM, int BN, int kFfmaBK>
__global__ void __launch_bounds__(kFfmaThreads)
    ffma_gemm_kernel(const T *__restrict__ A, const T *__restrict__ B, T *__restrict__ D,
                     DevLayout la, DevLayout lb, DevLayout ld, int64_t M, int64_t N, int64_t K, ErrCtx err)
{
#ifdef TMG_DEBUG_BOUNDS
    const int64_t a_limit = layout_extent(la), b_limit = layout_extent(lb), d_limit = layout_extent(ld);
#else
    const int64_t a_limit = 0, b_limit = 0, d_limit = 0;     // unused: the checks are constant true
#endif
    constexpr int TM = BM / 16, TN = BN / 16;
    constexpr int LA = BM * kFfmaBK / kFfmaThreads;     // elements of A each thread loads per slice
    constexpr int LB = BN * kFfmaBK / kFfmaThreads;
    __shared__ float As[2][kFfmaBK][BM + 1];
    __shared__ float Bs[2][kFfmaBK][BN + 1];

    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;

    float ra[LA], rb[LB];
    // element e = tid + 256 r of the slice: k fastest (row-major operands read
    // contiguous runs), then row
    auto load = [&](int64_t k0) {
#pragma unroll
        for (int r = 0; r < LA; ++r) {
            const int e = tid + kFfmaThreads * r;
            const int64_t m = m0 + e / kFfmaBK, k = k0 + e % kFfmaBK;
            const int64_t off = (m < M && k < K) ? crd2idx(la, m, k) : -1;
            ra[r] = (off >= 0 && bounds_ok(off, a_limit, err, kBndStoreD)) ? ld_elt(A, off) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < LB; ++r) {
            const int e = tid + kFfmaThreads * r;
            const int64_t n = n0 + e / kFfmaBK, k = k0 + e % kFfmaBK;
            const int64_t off = (n < N && k < K) ? crd2idx(lb, n, k) : -1;
            rb[r] = (off >= 0 && bounds_ok(off, b_limit, err, kBndStoreD)) ? ld_elt(B, off) : 0.f;
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int r = 0; r < LA; ++r) {
            const int e = tid + kFfmaThreads * r;
            As[buf][e % kFfmaBK][e / kFfmaBK] = ra[r];
        }
#pragma unroll
        for (int r = 0; r < LB; ++r) {
            const int e = tid + kFfmaThreads * r;
            Bs[buf][e % kFfmaBK][e / kFfmaBK] = rb[r];
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j)
            acc[i][j] = 0.f;

    load(0);
    stash(0);
    __syncthreads();
    int buf = 0;
    for (int64_t k0 = 0; k0 < K; k0 += kFfmaBK) {
        const bool more = k0 + kFfmaBK < K;
        if (more)
            load(k0 + kFfmaBK);
#pragma unroll
        for (int kk = 0; kk < kFfmaBK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i)
                a[i] = As[buf][kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < TN; ++j)
                b[j] = Bs[buf][kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j)
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more)
            stash(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t m = m0 + ty + 16 * i;
        if (m >= M)
            continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int64_t n = n0 + tx + 16 * j;
            if (n < N && bounds_ok(crd2idx(ld, m, n), d_limit, err, kBndStoreD))
                st_elt(D, crd2idx(ld, m, n), acc[i][j]);
        }
    }
}

// 16 bytes of T as fp32 values (exact for fp32 and bf16).
__device__ __forceinline__ void vec_to_f32(const uint4 &v, float (&f)[4])
{
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void vec_to_f32(const uint4 &v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Dense operands: A (M,K), B (N,K) and D (M,N) row-major (unit stride along
// the second coordinate), A and B rows 16-byte aligned, K a multiple of the
// 16-byte vector.  The tiles, thread map and k order are those of
// ffma_gemm_kernel (so the results are the same bits); the operands arrive
// as 16-byte vectors at plain row-major addresses.  A small problem runs
// this code once per thread and fetches it from L2 or DRAM as it goes, so
// its length is its time: the general kernel's per-element address
// arithmetic, straight-line, keeps the warps waiting on instruction fetch
// for several microseconds at 128^3.
template <typename T, int BM, int BN, int BK>
__global__ void __launch_bounds__(kFfmaThreads)
    ffma_dense_kernel(const T *__restrict__ A, const T *__restrict__ B, T *__restrict__ D, int64_t lda,
                      int64_t ldb, int64_t ldd, int M, int N, int K)
{
    constexpr int VEC = 16 / static_cast<int>(sizeof(T));
    constexpr int KV = BK / VEC;                          // vectors per tile row and K slice
    constexpr int NVA = BM * KV, NVB = BN * KV;
    constexpr int RA = (NVA + kFfmaThreads - 1) / kFfmaThreads, RB = (NVB + kFfmaThreads - 1) / kFfmaThreads;
    constexpr int TM = BM / 16, TN = BN / 16;
    __shared__ float As[2][BK][BM + 1];
    __shared__ float Bs[2][BK][BN + 1];

    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

    uint4 ra[RA], rb[RB];
    auto load = [&](int k0) {
#pragma unroll
        for (int r = 0; r < RA; ++r) {
            const int v = tid + kFfmaThreads * r, m = m0 + v / KV, k = k0 + (v % KV) * VEC;
            ra[r] = (v < NVA && m < M && k < K) ? __ldg(reinterpret_cast<const uint4 *>(A + m * lda + k))
                                                 : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int v = tid + kFfmaThreads * r, n = n0 + v / KV, k = k0 + (v % KV) * VEC;
            rb[r] = (v < NVB && n < N && k < K) ? __ldg(reinterpret_cast<const uint4 *>(B + n * ldb + k))
                                                 : make_uint4(0, 0, 0, 0);
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int r = 0; r < RA; ++r) {
            const int v = tid + kFfmaThreads * r;
            if (v < NVA) {
                float f[VEC];
                vec_to_f32(ra[r], f);
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    As[buf][(v % KV) * VEC + j][v / KV] = f[j];
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int v = tid + kFfmaThreads * r;
            if (v < NVB) {
                float f[VEC];
                vec_to_f32(rb[r], f);
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    Bs[buf][(v % KV) * VEC + j][v / KV] = f[j];
            }
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j)
            acc[i][j] = 0.f;

    load(0);
    stash(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < K; k0 += BK) {
        const bool more = k0 + BK < K;
        if (more)
            load(k0 + BK);
#pragma unroll 
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i)
                a[i] = As[buf][kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < TN; ++j)
                b[j] = Bs[buf][kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j)
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more)
            stash(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int m = m0 + ty + 16 * i;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int n = n0 + tx + 16 * j;
            if (m < M && n < N)
                st_elt(D, m * ldd + n, acc[i][j]);
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

template <typename T, int BM, int BN, int BK>
cudaError_t launch_ffma_cfg(const FfmaArgs &a, const ErrCtx &err, cudaStream_t s)
{
    dim3 grid(static_cast<unsigned>((a.N + BN - 1) / BN), static_cast<unsigned>((a.M + BM - 1) / BM));
    if (grid.y > 65535u)
        return cudaErrorInvalidConfiguration;
    // dense operands take the short kernel
    constexpr int64_t VEC = 16 / sizeof(T);
    const DevLayout &la = a.la, &lb = a.lb, &ld = a.ld;
    const bool dense = la.depth[0] == 1 && la.depth[1] == 1 && la.stride[1][0] == 1 && la.stride[0][0] % VEC == 0 &&
                       lb.depth[0] == 1 && lb.depth[1] == 1 && lb.stride[1][0] == 1 && lb.stride[0][0] % VEC == 0 &&
                       ld.depth[0] == 1 && ld.depth[1] == 1 && ld.stride[1][0] == 1 && a.K % VEC == 0 &&
                       (reinterpret_cast<uintptr_t>(a.A) & 15u) == 0 && (reinterpret_cast<uintptr_t>(a.B) & 15u) == 0 &&
                       a.M < (int64_t{1} << 31) && a.N < (int64_t{1} << 31) && a.K < (int64_t{1} << 31);
    if (dense) {
        note_launch();
        ffma_dense_kernel<T, BM, BN, BK><<<grid, kFfmaThreads, 0, s>>>(
            static_cast<const T *>(a.A), static_cast<const T *>(a.B), static_cast<T *>(a.D), la.stride[0][0],
            lb.stride[0][0], ld.stride[0][0], static_cast<int>(a.M), static_cast<int>(a.N), static_cast<int>(a.K));
        return cudaGetLastError();
    }
    note_launch();
    ffma_gemm_kernel<T, BM, BN, BK><<<grid, kFfmaThreads, 0, s>>>(static_cast<const T *>(a.A), static_cast<const T *>(a.B),
                                                                  static_cast<T *>(a.D), a.la, a.lb, a.ld, a.M, a.N, a.K,
                                                                  err);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_ffma_t(const FfmaArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    // Latency-bound small problems: many 16x16 tiles, 128-deep K slices (one
    // global round trip per 128 k); mid-size: 32x32; large: 64x64.
    const int64_t mn = a.M * a.N;
    if (mn <= static_cast<int64_t>(num_sms) * 16 * 16 * 2)
        return launch_ffma_cfg<T, 16, 16, 128>(a, err, s);
    if (mn <= static_cast<int64_t>(num_sms) * 64 * 64)
        return launch_ffma_cfg<T, 32, 32, 32>(a, err, s);
    return launch_ffma_cfg<T, 64, 64, 32>(a, err, s);
}

}  // namespace

cudaError_t launch_ffma(const FfmaArgs &a, int dtype, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    return dtype == 0 ? launch_ffma_t<float>(a, num_sms, err, s) : launch_ffma_t<__nv_bfloat16>(a, num_sms, err, s);
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
