// w4a8_skinny.cu — decode-shaped W4A8 GEMM (M <= 64): int8 activations A
// (M, K) x packed int4 weights B (N, K/2) -> exact int32 D (M, N), reading
// only the 4-bit weights from HBM.
//
// The pages' W4A8 kernel unpacks the int4 B to int8 in the kernel and uses
// an i8 x i8 -> i32 atom ("FlyDSL Kernel Authoring Skill", §10 item 10; §6
// integer WMMA rows).  GB300 has no integer tensor-core MMA, so here the
// unpack targets E4M3, which holds every int4 value exactly, and the MMA is
// tcgen05 kind::f8f6f4 with fp32 accumulation:
//   * each weight tile (128 rows of B x 128 k, 8 KB packed) lands in shared
//     memory by TMA; converter warps turn its nibbles into E4M3 bytes (a
//     16-entry lookup done with byte permutes) written in the 128-byte
//     swizzled K-major layout the MMA reads;
//   * an int8 activation a = 16 hi + lo with hi in [-8, 7] and lo in [0, 15],
//     both exact in E4M3: a small pre-pass writes A' (2 mp rows: hi rows,
//     then lo rows), and the MMA's N covers both (swap-AB as in skinny.cu:
//     the 128-row MMA dimension runs over weight rows);
//   * each fp32 column sum is an integer of magnitude <= 120 K < 2^22 for
//     K <= 32768, hence exact; the epilogue forms 16 S_hi + S_lo in int32.
// Work split, partial tiles and their fixed-order fix-up follow skinny.cu
// (stream-K over (tile, K block) units, per-tile counters per lane quarter).
//
// Warps: 0 TMA producer; 1 MMA issuer and TMEM owner; 2..5 epilogue (one
// per TMEM lane quarter); 6..13 converters.  Shared memory: a ring of
// STAGES staging slots (packed weights + A' tile), and a ring of kConvBufs
// converted weight tiles, each with its own barriers.
#include <cuda_bf16.h>

#include <cstring>

#include "internal.h"

namespace tmg {
namespace {

constexpr int kTileN = 128;                       // weight rows per tile (MMA M)
constexpr int kBK = 128;                          // k per K block: 128 E4M3 bytes per row
constexpr int kPackedBytes = kTileN * kBK / 2;    // 8 KB of int4 per tile and K block
constexpr int kConvBytes = kTileN * kBK;          // 16 KB of E4M3
constexpr int kConvBufs = 4;
constexpr int kMaxMP = 64;
constexpr int kConvWarps = 8;
constexpr int kThreads = 32 * (6 + kConvWarps);   // 448
constexpr int kTmemCols = 256;                    // two accumulators of up to 2 x 64 columns
constexpr int kMaxStages = 16;
constexpr int kSmemBudget = 225 * 1024;

// Staging slot: packed weights, then A' (2 mp rows x 128 bytes, 1 KB aligned).
__host__ __device__ constexpr int stage_bytes(int mp) { return kPackedBytes + 2 * mp * kBK; }
__host__ __device__ constexpr int conv_region() { return kConvBufs * kConvBytes; }
__host__ __device__ constexpr int bar_bytes() { return (2 * kMaxStages + 2 * kConvBufs + 4) * 8 + 16; }
int stages_for(int mp)
{
    int s = (kSmemBudget - conv_region() - bar_bytes() - 1024) / stage_bytes(mp);
    return s > kMaxStages ? kMaxStages : s;
}
int smem_for(int mp) { return stages_for(mp) * stage_bytes(mp) + conv_region() + bar_bytes() + 1024; }

__device__ __forceinline__ int64_t unit_start(int c, int64_t U, int G) { return (static_cast<int64_t>(c) * U) / G; }

__device__ __forceinline__ int seg_end(int kb0, int KB, int64_t left)
{
    return left < static_cast<int64_t>(KB - kb0) ? kb0 + static_cast<int>(left) : KB;
}

__device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int G)
{
    return static_cast<int>(((u + 1) * G - 1) / U);
}

// E4M3 codes of the int4 values: nibble n (two's complement) -> code.
// Non-negative v = 1..7 are (1 + m/8) 2^e with bias 7: 1 = 0x38, 2 = 0x40,
// 3 = 0x44, 4 = 0x48, 5 = 0x4A, 6 = 0x4C, 7 = 0x4E; -v sets the sign bit;
// -8 = -(1.0 x 2^3) = 0xD0.  Packed four per word, little-endian.
constexpr uint32_t kLut0 = 0x44403800u;   // n = 0..3  ->  0, 1, 2, 3
constexpr uint32_t kLut1 = 0x4E4C4A48u;   // n = 4..7  ->  4, 5, 6, 7
constexpr uint32_t kLut2 = 0xCACCCED0u;   // n = 8..11 -> -8, -7, -6, -5
constexpr uint32_t kLut3 = 0xB8C0C4C8u;   // n = 12..15 -> -4, -3, -2, -1

// Four nibbles (bits 0-15 of sel, nibble i -> output byte i) to four codes.
__device__ __forceinline__ uint32_t int4x4_to_e4m3(uint32_t sel)
{
    const uint32_t lo = __byte_perm(kLut0, kLut1, sel & 0x7777u);   // codes for n & 7, n < 8
    const uint32_t hi = __byte_perm(kLut2, kLut3, sel & 0x7777u);   // codes for n & 7, n >= 8
    const uint32_t pick = 0x3210u | (((sel >> 3) & 0x1111u) << 2);  // byte i from hi when n_i >= 8
    return __byte_perm(lo, hi, pick);
}

// Offset of 16-byte chunk j of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_offset(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }

// E4M3 codes of 0..15 (the low part of an activation): 0..7 as above, then
// 8..15 = (1 + m/8) 2^3 = 0x50..0x57.
constexpr uint32_t kLoLut2 = 0x53525150u;   // 8..11
constexpr uint32_t kLoLut3 = 0x57565554u;   // 12..15

__device__ __forceinline__ uint32_t uint4x4_to_e4m3(uint32_t sel)
{
    const uint32_t lo = __byte_perm(kLut0, kLut1, sel & 0x7777u);
    const uint32_t hi = __byte_perm(kLoLut2, kLoLut3, sel & 0x7777u);
    const uint32_t pick = 0x3210u | (((sel >> 3) & 0x1111u) << 2);
    return __byte_perm(lo, hi, pick);
}

// D[tmem] (+)= A[smem] . B[smem]^T, E4M3 operands, one CTA (kind::f8f6f4,
// K = 32 per instruction).
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// A' (2 mp rows x K, E4M3): row m < M holds the codes of hi = a >> 4, row
// mp + m those of lo = a & 15, for a = A[m, k]; padding rows are zero.  One
// thread per 4 consecutive k.
__global__ void split_activations_kernel(const int8_t *__restrict__ A, int M, int K, int mp, uint8_t *__restrict__ Ap)
{
    const int64_t words_per_row = K / 4;
    const int64_t total = 2 * static_cast<int64_t>(mp) * words_per_row;
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
         w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int rr = static_cast<int>(w / words_per_row);
        const int64_t k0 = (w % words_per_row) * 4;
        const bool lo_part = rr >= mp;
        const int m = lo_part ? rr - mp : rr;
        uint32_t out = 0;
        if (m < M) {
            uint32_t sel = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int a = A[static_cast<int64_t>(m) * K + k0 + i];
                const uint32_t nib = lo_part ? static_cast<uint32_t>(a & 15) : static_cast<uint32_t>((a >> 4) & 15);
                sel |= nib << (4 * i);
            }
            out = lo_part ? uint4x4_to_e4m3(sel) : int4x4_to_e4m3(sel);
        }
        *reinterpret_cast<uint32_t *>(Ap + static_cast<int64_t>(rr) * K + k0) = out;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    w4a8_skinny_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA,
                       int32_t *__restrict__ D, int64_t ldd, int M, int N, int K, int mp, int stages,
                       int32_t *__restrict__ partials, uint32_t *__restrict__ counters, ErrCtx err)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int sbytes = stage_bytes(mp);
    uint8_t *conv = smem + stages * sbytes;                   // kConvBufs x 16 KB
    uint64_t *full = reinterpret_cast<uint64_t *>(conv + conv_region());
    uint64_t *empty = full + kMaxStages;
    uint64_t *cready = empty + kMaxStages;                     // converted tile ready (converter warps)
    uint64_t *cfree = cready + kConvBufs;                      // converted tile consumed (MMA commit)
    uint64_t *tfull = cfree + kConvBufs;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int G = gridDim.x, c = blockIdx.x;
    const int tiles = (N + kTileN - 1) / kTileN;
    const int KB = K / kBK;                                    // K is a multiple of kBK
    const int64_t U = static_cast<int64_t>(tiles) * KB;
    const int64_t u_begin = unit_start(c, U, G), u_end = unit_start(c + 1, U, G);
    const uint32_t a_bytes = static_cast<uint32_t>(2 * mp * kBK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kConvBufs; ++b) {
            mbar_init(&cready[b], kConvWarps);
            mbar_init(&cfree[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmA);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------- TMA producer
            const uint64_t keep_a = policy_evict_last();    // A' is re-read by every CTA
            const uint64_t stream_b = policy_evict_first();  // the weights are read once
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t u = u_begin; u < u_end && ok;) {
                const int tile = static_cast<int>(u / KB);
                const int kb0 = static_cast<int>(u % KB);
                const int kb1 = seg_end(kb0, KB, u_end - u);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, err, abort_flag, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + stage * sbytes;
                    mbar_arrive_expect_tx(&full[stage], kPackedBytes + a_bytes);
                    tma_load_2d_hint(st, &tmB, &full[stage], kb * (kBK / 2), tile * kTileN, stream_b);
                    tma_load_2d_hint(st + kPackedBytes, &tmA, &full[stage], kb * kBK, 0, keep_a);
                    ++issued;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                u += kb1 - kb0;
            }
            for (int i = 0; i < stages && i < issued; ++i) {
                int s = stage - 1 - i;
                uint32_t ph = phase;
                if (s < 0) {
                    s += stages;
                    ph ^= 1u;
                }
                mbar_wait(&full[s], ph, err, nullptr, kSiteDrain);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            // MMA A = converted weights (128 rows), MMA B = A' (2 mp rows)
            const uint32_t idesc = idesc_e4m3_f32(kTileN, 2 * mp);
            int stage = 0, cb = 0, seg = 0;
            uint32_t phase = 0, cphase = 0;
            bool ok = true;
            for (int64_t u = u_begin; u < u_end && ok; ++seg) {
                const int kb0 = static_cast<int>(u % KB);
                const int kb1 = seg_end(kb0, KB, u_end - u);
                const int acc = seg & 1;
                if (!mbar_wait(&tempty[acc], ((seg >> 1) & 1) ^ 1u, err, abort_flag, kSiteMmaTmemEmpty))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * (kTmemCols / 2);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, err, abort_flag, kSiteMmaFull) ||
                        !mbar_wait(&cready[cb], cphase, err, abort_flag, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t wdesc = sdesc_kmajor_sw128(smem_u32(conv + cb * kConvBytes));
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(smem + stage * sbytes + kPackedBytes));
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k) {
                        const uint64_t koff = static_cast<uint64_t>((k * 32) >> 4);   // 32 bytes per MMA
                        mma_e4m3(d_tmem, wdesc + koff, adesc + koff, idesc, (kb != kb0) || (k != 0));
                    }
                    mma_commit(&empty[stage]);
                    mma_commit(&cfree[cb]);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++cb == kConvBufs) {
                        cb = 0;
                        cphase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit(&tfull[acc]);
                u += kb1 - kb0;
            }
        }
    } else if (warp >= 6) {
        // ------------------------------------------------- converters
        // Each K block: 128 rows x 64 bytes of nibbles -> 128 rows x 128
        // E4M3 bytes in the swizzled layout; a thread converts 16-byte
        // pieces (32 nibbles -> two 16-byte chunks of codes).
        const int ct = threadIdx.x - 6 * 32;
        int stage = 0, cb = 0;
        uint32_t phase = 0, cphase = 0;
        bool ok = true;
        for (int64_t u = u_begin; u < u_end && ok;) {
            const int kb0 = static_cast<int>(u % KB);
            const int kb1 = seg_end(kb0, KB, u_end - u);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(&full[stage], phase, err, abort_flag, kSiteMmaFull) ||
                    !mbar_wait(&cfree[cb], cphase ^ 1u, err, abort_flag, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = smem + stage * sbytes;
                uint8_t *dst = conv + cb * kConvBytes;
                for (int it = ct; it < kTileN * 4; it += kConvWarps * 32) {
                    const int r = it >> 2, p = it & 3;           // row, 32-k piece
                    const uint4 w = *reinterpret_cast<const uint4 *>(src + r * 64 + p * 16);
                    const uint4 c0 = make_uint4(int4x4_to_e4m3(w.x & 0xFFFFu), int4x4_to_e4m3(w.x >> 16),
                                                int4x4_to_e4m3(w.y & 0xFFFFu), int4x4_to_e4m3(w.y >> 16));
                    const uint4 c1 = make_uint4(int4x4_to_e4m3(w.z & 0xFFFFu), int4x4_to_e4m3(w.z >> 16),
                                                int4x4_to_e4m3(w.w & 0xFFFFu), int4x4_to_e4m3(w.w >> 16));
                    *reinterpret_cast<uint4 *>(dst + sw128_offset(r, 2 * p)) = c0;
                    *reinterpret_cast<uint4 *>(dst + sw128_offset(r, 2 * p + 1)) = c1;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&cready[cb]);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++cb == kConvBufs) {
                    cb = 0;
                    cphase ^= 1u;
                }
            }
            u += kb1 - kb0;
        }
    } else {
        // -------------------------------------------------- epilogue
        // thread owns weight row n_local = 32 q + lane; TMEM columns m and
        // mp + m hold the hi and lo sums of activation row m
        const int q = warp & 3;
        const int n_local = q * 32 + lane;
        int seg = 0;
        for (int64_t u = u_begin; u < u_end; ++seg) {
            const int tile = static_cast<int>(u / KB);
            const int kb0 = static_cast<int>(u % KB);
            const int kb1 = seg_end(kb0, KB, u_end - u);
            u += kb1 - kb0;
            const int acc = seg & 1;
            if (!mbar_wait(&tfull[acc], (seg >> 1) & 1, err, abort_flag, kSiteEpiTmemFull))
                break;
            tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * (kTmemCols / 2);
            int32_t v[kMaxMP];
#pragma unroll
            for (int ch = 0; ch < kMaxMP / 16; ++ch) {
                if (ch * 16 < mp) {
                    uint32_t h[16], l[16];
                    tmem_ld16(tb + ch * 16, h);
                    tmem_ld16(tb + mp + ch * 16, l);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[ch * 16 + j] = 16 * __float2int_rn(__uint_as_float(h[j])) + __float2int_rn(__uint_as_float(l[j]));
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[ch * 16 + j] = 0;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&tempty[acc]);

            const int n = tile * kTileN + n_local;
            if (kb0 == 0 && kb1 == KB) {
                if (n < N) {
#pragma unroll
                    for (int m = 0; m < kMaxMP; ++m)
                        if (m < M)
                            D[static_cast<int64_t>(m) * ldd + n] = v[m];
                }
                continue;
            }
            // Partial tile: integer partial sums; the last CTA to arrive for
            // (tile, quarter) adds them in CTA order and writes D.
            const int slot = 2 * c + (seg == 0 ? 0 : 1);
            int32_t *mine = partials + static_cast<int64_t>(slot) * mp * kTileN;
#pragma unroll
            for (int m = 0; m < kMaxMP; ++m)
                if (m < mp)
                    mine[m * kTileN + n_local] = v[m];
            __threadfence();
            __syncwarp();
            const int64_t t_first = static_cast<int64_t>(tile) * KB;
            const int c_first = unit_owner(t_first, U, G);
            const int c_last = unit_owner(t_first + KB - 1, U, G);
            uint32_t old = 0;
            if (lane == 0)
                old = atomicAdd(&counters[tile * 4 + q], 1u);
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == static_cast<uint32_t>(c_last - c_first)) {
                __threadfence();
                int32_t sum[kMaxMP];
#pragma unroll
                for (int m = 0; m < kMaxMP; ++m)
                    sum[m] = 0;
                // every contribution, this CTA's included, is read back from
                // scratch, so only one array of sums is live here
                for (int cc = c_first; cc <= c_last; ++cc) {
                    const int first_tile = static_cast<int>(unit_start(cc, U, G) / KB);
                    const int s2 = 2 * cc + (first_tile == tile ? 0 : 1);
                    const int32_t *p = partials + static_cast<int64_t>(s2) * mp * kTileN;
#pragma unroll
                    for (int m = 0; m < kMaxMP; ++m)
                        if (m < mp)
                            sum[m] += __ldcg(p + m * kTileN + n_local);
                }
                if (n < N) {
#pragma unroll
                    for (int m = 0; m < kMaxMP; ++m)
                        if (m < M)
                            D[static_cast<int64_t>(m) * ldd + n] = sum[m];
                }
                __syncwarp();
                if (lane == 0)
                    counters[tile * 4 + q] = 0;
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

int w4a8_skinny_grid(int64_t N, int64_t K, int num_sms)
{
    const int64_t units = ((N + kTileN - 1) / kTileN) * (K / kBK);
    return static_cast<int>(units < num_sms ? units : num_sms);
}

cudaError_t launch_w4a8_skinny(const W4a8SkinnyArgs &a, const ErrCtx &err, cudaStream_t s)
{
    // the activation split (one small launch), then the GEMM
    const int64_t words = 2 * static_cast<int64_t>(a.mp) * (a.K / 4);
    int64_t blocks = (words + 255) / 256;
    if (blocks > 1024)
        blocks = 1024;
    note_launch();
    split_activations_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const int8_t *>(a.A), a.M, a.K,
                                                                           a.mp, a.Ap);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int stages = stages_for(a.mp);
    const int smem = smem_for(a.mp);
    if ((e = ensure_smem_attr(reinterpret_cast<const void *>(w4a8_skinny_kernel), smem)) != cudaSuccess)
        return e;
    note_launch();
    w4a8_skinny_kernel<<<a.grid, kThreads, smem, s>>>(a.tmB, a.tmA, a.D, a.ldd, a.M, a.N, a.K, a.mp, stages,
                                                      a.partials, a.counters, err);
    return cudaGetLastError();
}

}  // namespace tmg
