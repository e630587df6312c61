// mxfp4.cu — block-scaled FP4 GEMM on tcgen05:
//   D (bf16, M x N) = A·Bᵀ, a(m,k) = e2m1(A code) * 2^(sA[m, k/32] - 127),
//   b(n,k) likewise, fp32 accumulation in tensor memory.
//
// The FlyDSL pages express this product with scaled MFMA/WMMA atoms whose
// E8M0 scales cover 32 consecutive K elements ("FlyDSL Kernel Authoring
// Skill", §6, "gfx1250 WMMA (wave32)": MX-scaled WMMA with block_size=32;
// "Kernel authoring guide", §4.3: the GFX950 scaled MFMA for MXFP4), and name
// an MXFP4 preshuffle GEMM kernel.  On sm_103a the product is one
// tcgen05.mma.kind::mxf4.block_scale.scale_vec::2X per 64 K elements
// (two scales per row per instruction), reading the packed e2m1 codes from
// 128-byte-swizzled shared memory and the scales from tensor memory.
//
// Per call, a small pre-pass (mx_scale_relayout_kernel) rewrites both
// scale arrays into the order the tensor core reads: for each 128-row block
// and each K block of 256 elements, 1 KB = two 512-byte chunks, chunk c
// holding K-blocks 4c..4c+3; inside a chunk, 16-byte line r0 (0..31) holds
// the four scales of rows r0, r0+32, r0+64, r0+96 for those K-blocks.
// Per K block of the main loop (128 bytes of codes per row):
//   producer lane   TMA of the A and B code tiles (128 x 128 bytes each)
//                   and two 1 KB bulk copies of the relaid scales, all
//                   completing on the stage's `full` barrier.
//   MMA lane        tcgen05.cp (32x128b, replicated to the four TMEM lane
//                   quarters) copies each scale chunk to this stage's TMEM
//                   scale columns; then four MMAs, each selecting its two
//                   scales inside the 32-bit column with the SF id (0 or 2).
//   epilogue warps  as in tc_bf16.cu.
// Tile 128 x 128, double-buffered accumulator (256 TMEM columns) plus
// 16 scale columns per stage.
#include <cuda_bf16.h>

#include "mx_common.cuh"

namespace tmg {
namespace {

using namespace mx;

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kStages = 6;
constexpr int kTileBytes = kBM * kBKBytes;   // 16 KB (A and B alike)
constexpr int kSfBytes = kSfBlock;      // 8 scales per row, 128 rows
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kAccCols = kBN;            // per buffer
constexpr int kSfCol0 = 2 * kAccCols;    // first scale column
constexpr int kSfColsPerStage = 16;      // A: 2 chunks x 4, B: 2 chunks x 4
constexpr int kGroupM = 8;
constexpr int kSmem = kStages * (2 * kTileBytes + 2 * kSfBytes) + (2 * kStages + 4) * 8 + 16 + 1024;

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &tm, int &tn)
{
    const int group = kGroupM * tiles_n;
    const int first_m = (t / group) * kGroupM;
    const int gm = min(tiles_m - first_m, kGroupM);
    const int r = t % group;
    tm = first_m + r % gm;
    tn = r / gm;
}

// Relayout pass: (rows, K/32) e8m0 row-major -> chunk order, rows grouped
// by `group_rows` (see mx_common.cuh).  One thread per 16-byte output line;
// blockIdx.y picks the operand.
struct RelayoutOperand {
    const uint8_t *S;
    uint8_t *out;
    int rows, group_rows, nsub;
    int wide;          // write the wide form (see mx_common.cuh)
};

// A CTA takes one 128-row sub-block and up to 8 consecutive K blocks: it
// reads the 128 x 64 bytes of scales row by row (8-byte loads, consecutive
// threads on consecutive bytes), then writes the 8 output blocks of 1 KB as
// consecutive 16-byte lines.  blockIdx.y picks the operand.
__global__ void __launch_bounds__(256)
    mx_scale_relayout_kernel(RelayoutOperand a, RelayoutOperand b, int sf_per_row, int num_kb)
{
    griddep_launch_dependents();
    const RelayoutOperand &o = blockIdx.y == 1 ? b : a;
    __shared__ uint32_t tile[128][17];                 // 16 words of scales per row, +1 pad
    const int kgroups = (num_kb + 7) / 8;
    const int64_t groups = (o.rows + o.group_rows - 1) / o.group_rows;
    const int64_t nblocks = groups * o.nsub * kgroups;
    for (int64_t blk = blockIdx.x; blk < nblocks; blk += gridDim.x) {
        const int kgrp = static_cast<int>(blk % kgroups);
        const int64_t rest = blk / kgroups;
        const int sub = static_cast<int>(rest % o.nsub);
        const int64_t g = rest / o.nsub;
        const int kb0 = kgrp * 8;
        const int nk = num_kb - kb0 < 8 ? num_kb - kb0 : 8;
        for (int e = threadIdx.x; e < 128 * 8; e += 256) {
            const int r = e >> 3, kk = e & 7;
            const int in_group = sub * 128 + r;
            const int64_t row = g * o.group_rows + in_group;
            uint2 v = make_uint2(0u, 0u);
            if (kk < nk && in_group < o.group_rows && row < o.rows)
                v = __ldg(reinterpret_cast<const uint2 *>(o.S + row * sf_per_row + (kb0 + kk) * 8));
            tile[r][2 * kk] = v.x;
            tile[r][2 * kk + 1] = v.y;
        }
        __syncthreads();
        const int reps = o.wide ? 4 : 1;
        for (int l = threadIdx.x; l < nk * 64 * reps; l += 256) {
            const int rep = l % reps, l1 = l / reps;
            const int kk = l1 >> 6, c = (l1 >> 5) & 1, r0 = l1 & 31;
            const int w = 2 * kk + c;
            const uint4 out = make_uint4(tile[r0][w], tile[32 + r0][w], tile[64 + r0][w], tile[96 + r0][w]);
            const int64_t blk = g * num_kb + kb0 + kk;
            uint8_t *dst;
            if (!o.wide) {
                dst = o.out + (blk * o.nsub + sub) * kSfBlock + c * kSfChunk + r0 * 16;
            } else {
                // copy p, half j: nsub == 1 -> (p, j) = (0, c); nsub == 2 -> (c, sub)
                const int p = o.nsub == 1 ? 0 : c;
                const int j = o.nsub == 1 ? c : sub;
                dst = o.out + blk * o.nsub * kWideSrcBytes + p * kWideSrcBytes + j * 2048 + rep * kSfChunk + r0 * 16;
            }
            *reinterpret_cast<uint4 *>(dst) = out;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    mxfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const uint8_t *__restrict__ relA, const uint8_t *__restrict__ relB,
                 __nv_bfloat16 *__restrict__ D, int M, int N, int K, int vec_ok, ErrCtx err)
{
    const int64_t d_limit = static_cast<int64_t>(M) * N;     // elements of D
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *tA = smem;                                   // kStages x 16 KB
    uint8_t *tB = tA + kStages * kTileBytes;              // kStages x 16 KB
    uint8_t *sfA = tB + kStages * kTileBytes;             // kStages x 1 KB
    uint8_t *sfB = sfA + kStages * kSfBytes;              // kStages x 1 KB
    uint64_t *full = reinterpret_cast<uint64_t *>(sfB + kStages * kSfBytes);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_kb = K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
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
        // ---------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            const uint8_t *sfa_src = relA + static_cast<int64_t>(tm) * num_kb * kSfBytes;
            const uint8_t *sfb_src = relB + static_cast<int64_t>(tn) * num_kb * kSfBytes;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait_warp(&empty[stage], phase ^ 1u, err, abort_flag, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_w(&full[stage], 2 * kTileBytes + 2 * kSfBytes);
                tma_load_2d_w(tA + stage * kTileBytes, &tmA, &full[stage], kb * kBKBytes, tm * kBM);
                tma_load_2d_w(tB + stage * kTileBytes, &tmB, &full[stage], kb * kBKBytes, tn * kBN);
                bulk_load_w(sfA + stage * kSfBytes, sfa_src + kb * kSfBytes, kSfBytes, &full[stage]);
                bulk_load_w(sfB + stage * kSfBytes, sfb_src + kb * kSfBytes, kSfBytes, &full[stage]);
                ++issued;
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        for (int i = 0; i < kStages && i < issued; ++i) {
            int s = stage - 1 - i;
            uint32_t ph = phase;
            if (s < 0) {
                s += kStages;
                ph ^= 1u;
            }
            mbar_wait(&full[s], ph, err, nullptr, kSiteDrain);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        // (the whole warp runs the loop; one elected lane issues)
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
            const int acc = local & 1;
            if (!mbar_wait_warp(&tempty[acc], ((local >> 1) & 1) ^ 1u, err, abort_flag, kSiteMmaTmemEmpty))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * kAccCols;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait_warp(&full[stage], phase, err, abort_flag, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sf_col = tmem_base + kSfCol0 + stage * kSfColsPerStage;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    tmem_cp_chunk_w(sf_col + c * 4,
                                    sdesc_noswizzle_rows16(smem_u32(sfA + stage * kSfBytes + c * kSfChunk)));
                    tmem_cp_chunk_w(sf_col + 8 + c * 4,
                                    sdesc_noswizzle_rows16(smem_u32(sfB + stage * kSfBytes + c * kSfChunk)));
                }
                const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(tA + stage * kTileBytes));
                const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(tB + stage * kTileBytes));
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // 64 codes = 32 bytes per MMA; scales (k/2) chunk, id 0 or 2
                    const uint64_t koff = static_cast<uint64_t>((k * 32) >> 4);
                    const int c = k >> 1;
                    const uint32_t id = (k & 1) ? 2u : 0u;
                    mma_mxf4_w(d_tmem, adesc + koff, bdesc + koff, idesc_mxf4(kBM, kBN, id),
                               sf_col + c * 4, sf_col + 8 + c * 4, (kb | k) != 0);
                }
                mma_commit_w(&empty[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            mma_commit_w(&tfull[acc]);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;
        int local = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            const int acc = local & 1;
            if (!mbar_wait(&tfull[acc], (local >> 1) & 1, err, abort_flag, kSiteEpiTmemFull))
                break;
            tc_fence_after();
            const int row = tm * kBM + q * 32 + lane;
            __nv_bfloat16 *drow = D + static_cast<int64_t>(row) * N;
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols + c * 32, v);
                const int col0 = tn * kBN + c * 32;
                const int64_t off = static_cast<int64_t>(row) * N + col0;
                if (row < M && span_ok(off, min(32, N - col0), d_limit, err, kBndStoreD)) {
                    if (vec_ok && col0 + 32 <= N) {
                        uint4 *dst = reinterpret_cast<uint4 *>(drow + col0);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
                            w.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
                            w.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
                            w.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
                            dst[j] = w;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < N)
                                drow[col0 + j] = __float2bfloat16_rn(__uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&tempty[acc]);
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

size_t mxfp4_relaid_scale_bytes(int64_t rows, int64_t K, int group_rows, bool wide)
{
    const int64_t groups = (rows + group_rows - 1) / group_rows;
    const int64_t nsub = (group_rows + 127) / 128;
    return static_cast<size_t>(groups * nsub * (K / kBK) * (wide ? kWideSrcBytes : kSfBlock));
}

cudaError_t launch_mx_scale_relayout(const uint8_t *sA, int M, uint8_t *relA, int groupA, const uint8_t *sB,
                                     int N, uint8_t *relB, int groupB, int K, bool wide, int num_sms,
                                     cudaStream_t s)
{
    const int num_kb = K / kBK;
    RelayoutOperand a{sA, relA, M, groupA, (groupA + 127) / 128, wide ? 1 : 0};
    RelayoutOperand b{sB, relB, N, groupB, (groupB + 127) / 128, wide ? 1 : 0};
    const int64_t kgroups = (num_kb + 7) / 8;
    const int64_t ba = (M + groupA - 1) / groupA * a.nsub * kgroups;
    const int64_t bb = (N + groupB - 1) / groupB * b.nsub * kgroups;
    int64_t blocks = ba > bb ? ba : bb;
    if (blocks > 8L * num_sms)
        blocks = 8L * num_sms;
    note_launch();
    mx_scale_relayout_kernel<<<dim3(static_cast<unsigned>(blocks), 2), 256, 0, s>>>(a, b, K / 32, num_kb);
    return cudaGetLastError();
}

cudaError_t launch_mxfp4(const Mxfp4Args &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(mxfp4_kernel), kSmem);
    if (e != cudaSuccess)
        return e;
    e = launch_mx_scale_relayout(a.sA, a.M, a.relA, kBM, a.sB, a.N, a.relB, kBN, a.K, false, num_sms, s);
    if (e != cudaSuccess)
        return e;
    const int tiles = ((a.M + kBM - 1) / kBM) * ((a.N + kBN - 1) / kBN);
    const int grid = tiles < num_sms ? tiles : num_sms;
    const int vec_ok = (a.N % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.D) & 15u) == 0);
    note_launch();
    mxfp4_kernel<<<grid, kThreads, kSmem, s>>>(a.tmA, a.tmB, a.relA, a.relB, static_cast<__nv_bfloat16 *>(a.D),
                                                a.M, a.N, a.K, vec_ok, err);
    return cudaGetLastError();
}

}  // namespace tmg
