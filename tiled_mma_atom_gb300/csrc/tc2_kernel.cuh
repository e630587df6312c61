// tc2_kernel.cuh — the GEMM kernel on CTA pairs: each cluster of two CTAs
// computes 256 x BN output tiles with tcgen05.mma.cta_group::2 (M = 256).
// CTA r (r = 0, 1) holds rows 128r..128r+127 of the A tile and rows
// r·BN/2 .. (r+1)·BN/2 - 1 of the B tile in its own shared memory, so each SM
// loads half the B tile it would need alone: per SM and K block, 16 KB of A
// plus BN/2 x 128 bytes of B instead of 16 KB plus BN x 128 bytes.
//
// Template parameters: the tile width BN; the input type IN (kInBf16:
// kind::f16, 64 elements per 128-byte K block; kInE4m3: kind::f8f6f4, 128
// elements per K block) — either way four 32-byte MMA steps per K block;
// and EPI, whether the fused epilogue runs (scale by row and column, bias by
// column, activation) before the bf16 rounding.
//
// Roles, in both CTAs unless stated:
//   warp 0        TMA producer for this CTA's halves; the loads of both CTAs
//                 complete on CTA 0's `full` barrier (CTA 0 announces the
//                 pair's byte count); waits on its own `empty` barrier.
//   warp 1        CTA 0 only: issues the pair MMAs and commits with a
//                 multicast arrive on the `empty` / `tmem_full` barriers of
//                 both CTAs.  Both CTAs' warp 1 allocate TMEM together.
//                 Warps 0 and 1 run their loops on all 32 lanes; one elected
//                 lane issues each copy, MMA and commit.
//   warps 2..     epilogue of this CTA's 128 accumulator rows (4 warps, or
//                 8 with the fused epilogue, two per lane quarter splitting
//                 the columns); each warp then arrives on CTA 0's
//                 `tmem_empty` barrier (count: the epilogue warps of both
//                 CTAs).
//
// Schedule (planned on the host by tc2_plan).  The tile width (256, 224,
// 192 or 128) and the schedule come from a cost model of measured per-K-block
// tile times: whole data-parallel waves (pair c takes tiles c, c + P, ...),
// or, where a partial last wave would leave most pairs idle, the last full
// wave and the partial one run stream-K — their (tile, K block) units cut
// into P equal contiguous runs, one per pair, each pair doing its run first.
// A tile split across pairs leaves fp32 partial sums in scratch; the last
// pair to finish a piece of it (a counter per tile, CTA and epilogue warp)
// adds the partials in pair order — a fixed order, so the result does not
// depend on timing — applies the epilogue, rounds to bf16 and resets the
// counter.  Tiles are visited in groups of group_m M-tiles.
//
// The fused epilogue follows the options of the preshuffle GEMM in "Kernel
// authoring guide", §11 "Complete example: Preshuffle GEMM" (scale_a,
// scale_b, bias; none / bias / bias_relu / bias_silu / bias_gelu), read as
// y = act(acc * scale_a[m] * scale_b[n] + bias[n]) with GELU in its erf form.
#pragma once

#include <cuda_bf16.h>

#include <cstring>

#include "internal.h"

namespace tmg {
namespace {

constexpr int kInBf16 = 0;
constexpr int kInE4m3 = 1;

constexpr int kBM = 256;           // rows per pair tile
constexpr int kHalfM = 128;        // rows per CTA
constexpr int kKBlockBytes = 128;  // bytes of each operand row per K block (one swizzle row)
// Warps: 0 producer, 1 MMA, then the epilogue warps — 4 (one per TMEM lane
// quarter) for the plain kernel, 8 (two per quarter, each taking half the
// columns) with the fused epilogue, whose arithmetic would otherwise pace
// the whole kernel.
__host__ __device__ constexpr int epi_warps(bool epi) { return epi ? 8 : 4; }
__host__ __device__ constexpr int tc2_threads(bool epi) { return 64 + 32 * epi_warps(epi); }

// Elements per K block for an input type.
__host__ __device__ constexpr int kb_elems(int in) { return in == kInE4m3 ? 128 : 64; }

// Shared memory, in order: the ring of A / B stages; the barriers; with the
// fused epilogue, per epilogue warp a copy of the scale_b and bias columns
// of its own chunks of the tile (copies of the whole tile's columns cost the
// 224-wide kernel its seventh stage: bf16 4096^3 with the fused epilogue
// but no operation took 78.5 instead of 76.5 us).  (The epilogue stores D straight from registers with 32-byte
// vector stores: staging tiles in shared memory for TMA stores was no faster
// and 16-byte stores wrote each 32-byte sector in halves — bf16 4096³:
// 83.5 -> 81.5 µs.)
template <int BN, bool EPI>
struct PairCfg {
    static constexpr int A_BYTES = kHalfM * kKBlockBytes;       // 16 KB
    static constexpr int B_BYTES = (BN / 2) * kKBlockBytes;     // this CTA's half
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // each epilogue warp's copy of the scale_b and bias columns of its own
    // chunks of the tile (the warps sharing a lane quarter split the chunks)
    static constexpr int COLW = EPI ? ((BN / 32 + epi_warps(EPI) / 4 - 1) / (epi_warps(EPI) / 4)) * 32 : 0;
    static constexpr int COLS_BYTES = epi_warps(EPI) * 2 * COLW * 4;
    static constexpr int RING_BUDGET = 220 * 1024 - 2048 - COLS_BYTES;
    static constexpr int STAGES = RING_BUDGET / STAGE_BYTES > 8 ? 8 : RING_BUDGET / STAGE_BYTES;
    static constexpr int TMEM_COLS = 512;
    static constexpr int BAR_BYTES = (2 * STAGES + 4) * 8 + 16;
    static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + COLS_BYTES + 1024;
};

// Operand majorness (template parameter MAJ): bit 0 set when A is MN-major
// (stored with M contiguous, i.e. Aᵀ row-major), bit 1 when B is (N
// contiguous).  bf16 only.  An MN-major operand's K block lands as 64 x 64
// boxes (64 M- or N-elements by 64 k, 128-byte swizzle): k row r of a box
// at r * 128 bytes, 8-row groups of 1024 bytes, the next 64 M/N elements in
// the next box 8 KB on — the canonical MN-major layout of the MMA, whose
// descriptor takes the 8 KB step between 64-element MN chunks as its
// leading byte offset and the 1 KB step between 8-row K groups as its
// stride byte offset.  One MMA (K = 16) covers 16 k rows = 2048 bytes.
constexpr int kMnBox = 64;
constexpr int kMnBoxBytes = kMnBox * kKBlockBytes;       // 8 KB
constexpr int kMnKStepBytes = 16 * kKBlockBytes;         // 2 KB per MMA

__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(kMnBoxBytes >> 4) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// kind::f16 instruction descriptor with the operands' transpose bits (bit 15
// A MN-major, bit 16 B MN-major).
__host__ __device__ constexpr uint32_t idesc_bf16_major(int M, int N, int maj)
{
    return idesc_bf16_f32(M, N) | ((maj & 1) ? (1u << 15) : 0u) | ((maj & 2) ? (1u << 16) : 0u);
}

// Tiles run in groups of group_m M-tiles, M-tile fastest within a group
// (the host's tc2_plan picks group_m).
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m, int &tm, int &tn)
{
    const int group = group_m * tiles_n;
    const int first_m = (t / group) * group_m;
    const int gm = min(tiles_m - first_m, group_m);
    const int r = t % group;
    tm = first_m + r % gm;
    tn = r / gm;
}

// Per-pair walk over its segments: its stream-K run first, then its
// data-parallel tiles, so the fix-ups of split tiles overlap the
// data-parallel work instead of trailing it.  The stream-K tiles are the
// first sk_tiles of the grouped order and the data-parallel ones follow, so
// the pairs sweep the grouped order front to back (operand panels stay in
// L2 while they are used).  Every role of both CTAs walks the same sequence.
struct SegWalk {
    int nclusters, dp_tiles, sk_tiles, num_kb;
    int64_t u, u_end;          // stream-K units of this pair (relative to the stream-K region)
    int next_dp;               // next data-parallel tile
    int sk_seg;                // stream-K segments handed out so far

    __device__ SegWalk(int c, int nc, int dp, int sk, int nkb) : nclusters(nc), dp_tiles(dp), sk_tiles(sk), num_kb(nkb)
    {
        const int64_t U = static_cast<int64_t>(sk) * nkb;
        u = U * c / nc;
        u_end = U * (c + 1) / nc;
        next_dp = c;
        sk_seg = 0;
    }

    // Next segment: tile, K-block range, whether it is a piece of a split
    // tile, and the pair's scratch slot for it (0 = first piece, 1 = last).
    __device__ bool next(int &tile, int &kb0, int &kb1, bool &partial, int &slot)
    {
        if (u >= u_end) {
            if (next_dp >= dp_tiles)
                return false;
            tile = sk_tiles + next_dp;
            next_dp += nclusters;
            kb0 = 0;
            kb1 = num_kb;
            partial = false;
            slot = 0;
            return true;
        }
        const int rel = static_cast<int>(u / num_kb);
        kb0 = static_cast<int>(u % num_kb);
        const int64_t left = u_end - u;
        kb1 = left < static_cast<int64_t>(num_kb - kb0) ? kb0 + static_cast<int>(left) : num_kb;
        tile = rel;
        partial = !(kb0 == 0 && kb1 == num_kb);
        slot = sk_seg == 0 ? 0 : 1;
        ++sk_seg;
        u += kb1 - kb0;
        return true;
    }
};

// Pair whose stream-K run contains unit u (of U units over P pairs).
__device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int P)
{
    return static_cast<int>(((u + 1) * P - 1) / U);
}

// Round 32 fp32 values of one output row to bf16 and store them at
// drow[col0 .. col0+31] (bounded by N): two 32-byte stores (whole sectors)
// where the row segment starts on a 32-byte boundary, else four 16-byte
// stores (vec_ok: 16-byte aligned rows), else one by one.
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16 *drow, int col0, int N, int vec_ok,
                                                const float (&v)[32])
{
    if (vec_ok && col0 + 32 <= N && (reinterpret_cast<uintptr_t>(drow + col0) & 31u) == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
            st_global_v8(drow + col0 + 16 * j, pack_bf16x2(v[16 * j + 0], v[16 * j + 1]),
                         pack_bf16x2(v[16 * j + 2], v[16 * j + 3]), pack_bf16x2(v[16 * j + 4], v[16 * j + 5]),
                         pack_bf16x2(v[16 * j + 6], v[16 * j + 7]), pack_bf16x2(v[16 * j + 8], v[16 * j + 9]),
                         pack_bf16x2(v[16 * j + 10], v[16 * j + 11]), pack_bf16x2(v[16 * j + 12], v[16 * j + 13]),
                         pack_bf16x2(v[16 * j + 14], v[16 * j + 15]));
    } else if (vec_ok && col0 + 32 <= N) {
        uint4 *dst = reinterpret_cast<uint4 *>(drow + col0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 w;
            w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
            w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
            w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
            w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
            dst[j] = w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < N)
                drow[col0 + j] = __float2bfloat16_rn(v[j]);
    }
}

// 32 integer-valued fp32 results of one row as int32 at drow[col0 ..]
// (bounded by N), stored or added to what D holds (the W4A8 GEMM's K
// segments).  The values are exact integers, so rounding is exact.
__device__ __forceinline__ void store_row_i32(int32_t *drow, int col0, int N, int vec_ok, const float (&v)[32],
                                              bool accumulate)
{
    if (vec_ok && col0 + 32 <= N) {
        int4 *dst = reinterpret_cast<int4 *>(drow + col0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int4 o = accumulate ? dst[j] : make_int4(0, 0, 0, 0);
            o.x += __float2int_rn(v[4 * j]);
            o.y += __float2int_rn(v[4 * j + 1]);
            o.z += __float2int_rn(v[4 * j + 2]);
            o.w += __float2int_rn(v[4 * j + 3]);
            dst[j] = o;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < N)
                drow[col0 + j] = (accumulate ? drow[col0 + j] : 0) + __float2int_rn(v[j]);
    }
}

// GELU(y) = y * Phi(y), Phi(y) = erfc(-y / sqrt 2) / 2, with erfc from
// Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26:
// erfc(x) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) e^(-x^2),
// t = 1 / (1 + p x), x >= 0, |error| <= 1.5e-7 — far below the bf16 rounding
// of the result.  For y < 0, Phi(y) = erfc(|y| / sqrt 2) / 2 directly (no
// cancellation); for y >= 0, 1 minus that.
__device__ __forceinline__ float gelu_as(float y)
{
    const float x = fabsf(y) * 0.70710678118654752f;
    const float t = __fdividef(1.f, fmaf(0.3275911f, x, 1.f));
    const float poly =
        t * fmaf(fmaf(fmaf(fmaf(1.061405429f, t, -1.453152027f), t, 1.421413741f), t, -0.284496736f), t,
                 0.254829592f);
    const float half_erfc = 0.5f * poly * __expf(-x * x);
    return y * (y >= 0.f ? 1.f - half_erfc : half_erfc);
}

// The fused epilogue on 32 consecutive outputs of one row:
// v[j] <- act(v[j] * sa_row * sb[col0+j] + bias[col0+j]).  `cols` is the
// warp's shared-memory copy of the tile's scale_b and bias columns (staged
// once per tile, zeros past N), read as broadcasts.  Every branch is uniform
// across the warp and sits outside the per-element loops, so each step is
// one short unrolled loop and the code a warp runs stays small (a switch
// inside the 32-way unrolled loop made the epilogue code large enough to
// slow the whole kernel 2-4x).  SiLU uses the fast exponential and division
// intrinsics, GELU the erfc formula above: their errors (a few fp32 ulp,
// 1.5e-7) are far below the bf16 rounding that follows.
template <int COLW>
__device__ __forceinline__ void apply_epilogue(float (&v)[32], const Tc2Epi &e, float sa_row, const float *cols,
                                               int cl)
{
    if (e.scale_a) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            v[j] *= sa_row;
    }
    if (e.scale_b) {
        const float4 *w = reinterpret_cast<const float4 *>(cols + cl);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 t = w[j];
            v[4 * j] *= t.x;
            v[4 * j + 1] *= t.y;
            v[4 * j + 2] *= t.z;
            v[4 * j + 3] *= t.w;
        }
    }
    if (e.epi >= kEpiBias) {
        const float4 *w = reinterpret_cast<const float4 *>(cols + COLW + cl);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 t = w[j];
            v[4 * j] += t.x;
            v[4 * j + 1] += t.y;
            v[4 * j + 2] += t.z;
            v[4 * j + 3] += t.w;
        }
    }
    if (e.epi == kEpiBiasRelu) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            v[j] = fmaxf(v[j], 0.f);
    } else if (e.epi == kEpiBiasSilu) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            v[j] = __fdividef(v[j], 1.f + __expf(-v[j]));
    } else if (e.epi == kEpiBiasGelu) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            v[j] = gelu_as(v[j]);
    }
}

template <int BN, int IN, bool EPI, int MAJ = 0>
__global__ void __launch_bounds__(tc2_threads(EPI), 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    __nv_bfloat16 *__restrict__ D, int64_t ldd, int M, int N, int K, int dp_tiles, int sk_tiles,
                    int group_m, float *__restrict__ partials, uint32_t *__restrict__ counters, int vec_ok, Tc2Epi epi,
                    ErrCtx err)
{
    using C = PairCfg<BN, EPI>;
    static_assert(MAJ == 0 || (IN == kInBf16 && !EPI && ((MAJ & 2) == 0 || (BN / 2) % kMnBox == 0)),
                  "MN-major operands: plain bf16; an MN-major B needs whole 64-column boxes per CTA");
    const int64_t d_limit = static_cast<int64_t>(M - 1) * ldd + N;     // elements of D
    constexpr int KB_ELEMS = kb_elems(IN);
    constexpr int STAGES = C::STAGES;
    constexpr uint32_t STAGE_TX = 2u * C::STAGE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * C::A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * C::STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *epi_cols = reinterpret_cast<float *>(smem + STAGES * C::STAGE_BYTES + C::BAR_BYTES);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + BN - 1) / BN;
    const int num_kb = (K + KB_ELEMS - 1) / KB_ELEMS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 2 * epi_warps(EPI));
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();          // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------- TMA producer
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        SegWalk walk(cluster, nclusters, dp_tiles, sk_tiles, num_kb);
        int tile, kb0, kb1, slot;
        bool partial;
        while (ok && walk.next(tile, kb0, kb1, partial, slot)) {
            int tm, tn;
            tile_coords(tile, tiles_m, tiles_n, group_m, tm, tn);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_cluster_warp(&empty[stage], phase ^ 1u, err, abort_flag, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                if (rank == 0)
                    mbar_arrive_expect_tx_w(&full[stage], STAGE_TX);
                const uint32_t bar0 = mapa_shared(smem_u32(&full[stage]), 0);
                const int a_row = tm * kBM + rank * kHalfM, b_row = tn * BN + rank * (BN / 2);
                if constexpr (MAJ & 1) {
#pragma unroll
                    for (int j = 0; j < kHalfM / kMnBox; ++j)
                        tma_load_2d_pair_w(sA + stage * C::A_BYTES + j * kMnBoxBytes, &tmA, bar0, a_row + j * kMnBox,
                                           kb * KB_ELEMS);
                } else {
                    tma_load_2d_pair_w(sA + stage * C::A_BYTES, &tmA, bar0, kb * KB_ELEMS, a_row);
                }
                if constexpr ((MAJ & 2) != 0) {
#pragma unroll
                    for (int j = 0; j < (BN / 2) / kMnBox; ++j)
                        tma_load_2d_pair_w(sB + stage * C::B_BYTES + j * kMnBoxBytes, &tmB, bar0, b_row + j * kMnBox,
                                           kb * KB_ELEMS);
                } else {
                    tma_load_2d_pair_w(sB + stage * C::B_BYTES, &tmB, bar0, kb * KB_ELEMS, b_row);
                }
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Tail: wait until the MMA has released every stage this CTA
        // filled (so no multicast arrive is still on its way here), and
        // in CTA 0 until every load of the pair has landed.
        for (int i = 0; i < STAGES && i < issued; ++i) {
            int s = stage - 1 - i;
            uint32_t ph = phase;
            if (s < 0) {
                s += STAGES;
                ph ^= 1u;
            }
            if (rank == 0)
                mbar_wait_cluster(&full[s], ph, err, abort_flag, kSiteDrain);
            mbar_wait_cluster(&empty[s], ph, err, abort_flag, kSiteDrain);
        }
    } else if (warp == 1) {
        if (rank == 0) {
            // -------------------------------------------- MMA issuer
            // (the whole warp runs the loop; one elected lane issues)
            constexpr uint32_t idesc = IN == kInE4m3 ? idesc_e4m3_f32(kBM, BN) : idesc_bf16_major(kBM, BN, MAJ);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            SegWalk walk(cluster, nclusters, dp_tiles, sk_tiles, num_kb);
            int tile, kb0, kb1, slot;
            bool partial;
            while (ok && walk.next(tile, kb0, kb1, partial, slot)) {
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                ++local;
                if (!mbar_wait_cluster_warp(&tempty[acc], acc_phase ^ 1u, err, abort_flag, kSiteMmaTmemEmpty))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait_cluster_warp(&full[stage], phase, err, abort_flag, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = smem_u32(sA + stage * C::A_BYTES), b_s = smem_u32(sB + stage * C::B_BYTES);
                    const uint64_t adesc = (MAJ & 1) ? sdesc_mnmajor_sw128(a_s) : sdesc_kmajor_sw128(a_s);
                    const uint64_t bdesc = (MAJ & 2) ? sdesc_mnmajor_sw128(b_s) : sdesc_kmajor_sw128(b_s);
                    // per MMA: 32 bytes along a K-major row, or 16 k rows of an MN-major box
                    constexpr uint64_t astep = ((MAJ & 1) ? kMnKStepBytes : 32) >> 4;
                    constexpr uint64_t bstep = ((MAJ & 2) ? kMnKStepBytes : 32) >> 4;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if constexpr (IN == kInE4m3)
                            mma_e4m3_pair_w(d_tmem, adesc + k * astep, bdesc + k * bstep, idesc, (kb != kb0) || (k != 0));
                        else
                            mma_bf16_pair_w(d_tmem, adesc + k * astep, bdesc + k * bstep, idesc, (kb != kb0) || (k != 0));
                    }
                    mma_commit_pair_w(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit_pair_w(&tfull[acc], 0x3);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        constexpr int NEPI = epi_warps(EPI);
        // 32-column chunks per warp: the warps sharing a lane quarter split
        // the tile's BN / 32 chunks, the first ones taking one more when
        // the count is odd (224-wide tiles: 4 + 3)
        constexpr int CHUNKS = (BN / 32 + NEPI / 4 - 1) / (NEPI / 4);
        const int e = warp - 2;                          // epilogue warp index
        const int q = warp & 3;                          // its TMEM lane quarter
        const int c_begin = (e / 4) * CHUNKS, c_end = min(BN / 32, c_begin + CHUNKS);
        const int64_t U = static_cast<int64_t>(sk_tiles) * num_kb;
        int local = 0;
        SegWalk walk(cluster, nclusters, dp_tiles, sk_tiles, num_kb);
        int tile, kb0, kb1, slot;
        bool partial;
        while (walk.next(tile, kb0, kb1, partial, slot)) {
            int tm, tn;
            tile_coords(tile, tiles_m, tiles_n, group_m, tm, tn);
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            ++local;
            const int row = tm * kBM + static_cast<int>(rank) * kHalfM + q * 32 + lane;
            // this warp's copy of the tile's scale_b / bias columns, staged
            // while the accumulator is still being computed
            float *cols = epi_cols + e * 2 * C::COLW;
            float sa_row = 1.f;
            if constexpr (EPI) {
                if (epi.scale_a && row < M)
                    sa_row = __ldg(epi.scale_a + row);
                __syncwarp();            // the previous tile's reads are done
                const int c0 = tn * BN;
                if (epi.scale_b)
                    for (int i = c_begin * 32 + lane; i < c_end * 32; i += 32)
                        cols[i - c_begin * 32] = c0 + i < N ? __ldg(epi.scale_b + c0 + i) : 0.f;
                if (epi.epi >= kEpiBias)
                    for (int i = c_begin * 32 + lane; i < c_end * 32; i += 32)
                        cols[C::COLW + i - c_begin * 32] = c0 + i < N ? __ldg(epi.bias + c0 + i) : 0.f;
                __syncwarp();
            }
            if (!mbar_wait_cluster(&tfull[acc], acc_phase, err, abort_flag, kSiteEpiTmemFull))
                break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            __nv_bfloat16 *drow = D + static_cast<int64_t>(row) * ldd;
            if (!partial) {
#pragma unroll 1
                for (int c = c_begin; c < c_end; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tbase + c * 32, r);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = __uint_as_float(r[j]);
                    if constexpr (EPI)
                        apply_epilogue<C::COLW>(v, epi, sa_row, cols, (c - c_begin) * 32);
                    const int col0 = tn * BN + c * 32;
                    if constexpr (EPI) {
                        if (epi.out_i32) {
                            if (row < M && span_ok(static_cast<int64_t>(row) * ldd + col0, min(32, N - col0), d_limit,
                                                   err, kBndStoreD))
                                store_row_i32(reinterpret_cast<int32_t *>(D) + static_cast<int64_t>(row) * ldd, col0, N,
                                              vec_ok, v, epi.out_i32 == 2);
                            continue;
                        }
                    }
                    if (row < M && span_ok(static_cast<int64_t>(row) * ldd + col0, min(32, N - col0), d_limit, err,
                                           kBndStoreD))
                        store_row_chunk(drow, col0, N, vec_ok, v);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
                continue;
            }
            // Piece of a split tile: this warp's 32 rows x BN columns go to
            // scratch, laid out [chunk][4-column group][lane][4] so each
            // store moves 512 contiguous bytes.
            const int64_t warp_elems = 32 * BN;
            const int64_t p_limit = static_cast<int64_t>(nclusters) * 2 * 2 * 4 * warp_elems;   // floats of scratch
            const int64_t mine_off = ((static_cast<int64_t>(2 * cluster + slot) * 2 + rank) * 4 + q) * warp_elems;
            float *mine = partials + mine_off;
#pragma unroll 1
            for (int c = c_begin; c < c_end; ++c) {
                uint32_t r[32];
                tmem_ld32(tbase + c * 32, r);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (span_ok(mine_off + ((c * 8 + j) * 32 + lane) * 4, 4, p_limit, err, kBndPartials))
                        reinterpret_cast<float4 *>(mine)[(c * 8 + j) * 32 + lane] =
                            make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
            __threadfence();
            __syncwarp();
            const int rel = tile;
            const int c_first = unit_owner(static_cast<int64_t>(rel) * num_kb, U, nclusters);
            const int c_last = unit_owner(static_cast<int64_t>(rel + 1) * num_kb - 1, U, nclusters);
            const int64_t counter_idx = (static_cast<int64_t>(rel) * 2 + rank) * NEPI + e;
            if (!bounds_ok(counter_idx, static_cast<int64_t>(sk_tiles) * 2 * NEPI, err, kBndCounters))
                continue;
            uint32_t *counter = counters + counter_idx;
            uint32_t old = 0;
            if (lane == 0)
                old = atomicAdd(counter, 1u);
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old != static_cast<uint32_t>(c_last - c_first))
                continue;
            // last to arrive: add the pieces in pair order, round, store
            __threadfence();
#pragma unroll 1
            for (int c = c_begin; c < c_end; ++c) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = 0.f;
                for (int cc = c_first; cc <= c_last; ++cc) {
                    const int first_tile = static_cast<int>((U * cc / nclusters) / num_kb);
                    const int s2 = first_tile == tile ? 0 : 1;
                    const int64_t src_off = ((static_cast<int64_t>(2 * cc + s2) * 2 + rank) * 4 + q) * warp_elems;
                    const float4 *src = reinterpret_cast<const float4 *>(partials + src_off);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (!span_ok(src_off + ((c * 8 + j) * 32 + lane) * 4, 4, p_limit, err, kBndPartials))
                            continue;
                        const float4 p = __ldcg(src + (c * 8 + j) * 32 + lane);
                        v[4 * j] += p.x;
                        v[4 * j + 1] += p.y;
                        v[4 * j + 2] += p.z;
                        v[4 * j + 3] += p.w;
                    }
                }
                if constexpr (EPI) {
                    apply_epilogue<C::COLW>(v, epi, sa_row, cols, (c - c_begin) * 32);
                    if (epi.out_i32) {
                        if (row < M && span_ok(static_cast<int64_t>(row) * ldd + tn * BN + c * 32,
                                               min(32, N - tn * BN - c * 32), d_limit, err, kBndStoreD))
                            store_row_i32(reinterpret_cast<int32_t *>(D) + static_cast<int64_t>(row) * ldd,
                                          tn * BN + c * 32, N, vec_ok, v, epi.out_i32 == 2);
                        continue;
                    }
                }
                if (row < M && span_ok(static_cast<int64_t>(row) * ldd + tn * BN + c * 32, min(32, N - tn * BN - c * 32),
                                       d_limit, err, kBndStoreD))
                    store_row_chunk(drow, tn * BN + c * 32, N, vec_ok, v);
            }
            __syncwarp();
            if (lane == 0)
                *counter = 0;
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();          // no CTA leaves while its peer may still touch it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int IN, bool EPI, int MAJ = 0>
cudaError_t launch_pair(const TcArgs &a, const Tc2Epi &epi, const ErrCtx &err, cudaStream_t s)
{
    using C = PairCfg<BN, EPI>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    static_assert(C::STAGES >= 4, "pipeline depth");
    static_assert(2 * BN <= C::TMEM_COLS, "TMEM budget");
    static_assert(C::B_BYTES % 1024 == 0, "B half must be whole 8-row swizzle atoms");
    if (a.group_m < 1)          // tc2_plan not called
        return cudaErrorInvalidValue;
    auto kern = tc2_gemm_kernel<BN, IN, EPI, MAJ>;
    constexpr int SMEM = C::SMEM;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), SMEM);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * a.pairs);
    cfg.blockDim = dim3(tc2_threads(EPI));
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int vec_ok = (a.ldd % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.D) & 15u) == 0);
    note_launch();
    e = cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, static_cast<__nv_bfloat16 *>(a.D), a.ldd, a.M, a.N, a.K,
                           a.dp_tiles, a.sk_tiles, a.group_m, a.partials, a.counters, vec_ok, epi, err);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace
}  // namespace tmg
