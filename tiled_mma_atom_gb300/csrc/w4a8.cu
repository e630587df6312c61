// w4a8.cu — the operand side of the W4A8 GEMM (int8 A x packed int4 B,
// exact int32 result).
//
// The pages' W4A8 GEMM ("FlyDSL Kernel Authoring Skill", §10
// Troubleshooting, item 10) unpacks the int4 B to int8 in the kernel and
// multiplies with an i8 x i8 -> i32 MMA atom (§6).  GB300 has no integer
// tensor-core MMA (tcgen05 kind::i8 is not available on sm_103a), so here
// both operands are unpacked to bf16 — every int8 and int4 value is exact in
// bf16 — and the product runs on the bf16 tensor cores with fp32
// accumulation, which is exact for integer sums below 2^24: the library
// cuts K into segments of at most 8192 (|sum| <= 1024 * 8192 = 2^23) and the
// GEMM epilogue stores or adds each segment's result into the int32 D
// (api.cu, gemm_w4a8_impl).
//
// unpack: P[r * ldp + k] = bf16(X(r, k)) for k < K, 0 for K <= k < ldp, with
// X either int8 (X(r, k) = A[r * K + k]) or packed int4 (two's complement
// nibbles, the even k in the low nibble of byte r * K/2 + k/2, or of the
// pre-shuffled image's byte holding (r, k)).  Each thread
// converts 8 consecutive k: 8 bytes of int8 or 4 bytes of int4 in, 16 bytes
// of bf16 out.  HBM-bound.
#include <cuda_bf16.h>

#include "internal.h"

namespace tmg {
namespace {

constexpr int kUnpackThreads = 256;

__device__ __forceinline__ uint32_t bf16x2_of_ints(int lo, int hi)
{
    // small integers convert exactly; pack_bf16x2 rounds to nearest even,
    // which keeps them unchanged
    return pack_bf16x2(static_cast<float>(lo), static_cast<float>(hi));
}

__device__ __forceinline__ int int4_at(uint32_t word, int j)   // nibble j (0..7) of a 32-bit word
{
    return static_cast<int>(static_cast<int32_t>(word << (28 - 4 * j)) >> 28);
}

// SHUF: X is the pre-shuffled int4 image (K a multiple of 32, so a group
// of 8 k is either whole or entirely past K).
template <bool INT4, bool SHUF = false>
__global__ void __launch_bounds__(kUnpackThreads)
    unpack_kernel(const uint8_t *__restrict__ X, int64_t rows, int64_t K, uint16_t *__restrict__ P, int64_t ldp,
                  int vec_ok)
{
    const int64_t groups_per_row = ldp / 8;
    const int64_t total = rows * groups_per_row;
    const int64_t KB = (K + kW4BK - 1) / kW4BK;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = g / groups_per_row;
        const int64_t k0 = (g % groups_per_row) * 8;
        int v[8];
        if constexpr (SHUF) {
            const uint32_t w =
                k0 < K ? *reinterpret_cast<const uint32_t *>(X + w4a8_preshuffled_offset(r, k0, KB)) : 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = int4_at(w, j);
        } else if (vec_ok && k0 + 8 <= K) {
            if constexpr (INT4) {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(X + r * (K / 2) + k0 / 2);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v[j] = int4_at(w, j);
            } else {
                const uint2 w = *reinterpret_cast<const uint2 *>(X + r * K + k0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[j] = static_cast<int8_t>((w.x >> (8 * j)) & 0xFF);
                    v[4 + j] = static_cast<int8_t>((w.y >> (8 * j)) & 0xFF);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t k = k0 + j;
                if (k >= K) {
                    v[j] = 0;
                } else if constexpr (INT4) {
                    const uint8_t b = X[r * (K / 2) + k / 2];
                    v[j] = int4_at(static_cast<uint32_t>((k & 1) ? (b >> 4) : (b & 0x0F)), 0);
                } else {
                    v[j] = static_cast<int8_t>(X[r * K + k]);
                }
            }
        }
        *reinterpret_cast<uint4 *>(P + r * ldp + k0) = make_uint4(bf16x2_of_ints(v[0], v[1]), bf16x2_of_ints(v[2], v[3]),
                                                                  bf16x2_of_ints(v[4], v[5]), bf16x2_of_ints(v[6], v[7]));
    }
}

unsigned grid_for(int64_t work, int num_sms)
{
    const int64_t blocks = (work + kUnpackThreads - 1) / kUnpackThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    return static_cast<unsigned>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

cudaError_t launch_unpack_w4a8(const void *A, const void *B, int64_t M, int64_t N, int64_t K, void *PA, void *PB,
                               int64_t ldp, int num_sms, cudaStream_t s, bool b_preshuffled)
{
    const uintptr_t pa = reinterpret_cast<uintptr_t>(A), pb = reinterpret_cast<uintptr_t>(B);
    const int vec_a = (K % 8 == 0) && (pa % 8 == 0);
    const int vec_b = (K % 8 == 0) && (pb % 4 == 0);
    note_launch();
    unpack_kernel<false><<<grid_for(M * (ldp / 8), num_sms), kUnpackThreads, 0, s>>>(
        static_cast<const uint8_t *>(A), M, K, static_cast<uint16_t *>(PA), ldp, vec_a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    note_launch();
    if (b_preshuffled)
        unpack_kernel<true, true><<<grid_for(N * (ldp / 8), num_sms), kUnpackThreads, 0, s>>>(
            static_cast<const uint8_t *>(B), N, K, static_cast<uint16_t *>(PB), ldp, 1);
    else
        unpack_kernel<true><<<grid_for(N * (ldp / 8), num_sms), kUnpackThreads, 0, s>>>(
            static_cast<const uint8_t *>(B), N, K, static_cast<uint16_t *>(PB), ldp, vec_b);
    return cudaGetLastError();
}

}  // namespace tmg
