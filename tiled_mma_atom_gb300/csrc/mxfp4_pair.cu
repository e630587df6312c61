// mxfp4_pair.cu — the MXFP4 GEMM of mxfp4.cu on CTA pairs
// (tcgen05.mma.cta_group::2.kind::mxf4.block_scale, M = 256).
//
// Each cluster of two CTAs computes a 256 x BN tile (BN = 256, 192 or 128).  CTA r
// keeps in its own shared memory rows 128r..128r+127 of the A codes, rows
// r·BN/2.. of the B codes, the scales of its own 128 A rows and the scales
// of all BN B rows (its tensor core multiplies its 128 rows by every column
// of the tile, so it needs every B scale).  All four loads of both CTAs are
// TMA copies completing on CTA 0's barriers: the codes on `full`, the scales
// on `sfull`.  Warp roles: 0 TMA producer; 1 MMA issuer (CTA 0); 2 scale
// copier (CTA 0), which moves each stage's scales of both CTAs into their
// TMEM with tcgen05.cp.cta_group::2 copies and commits to the stage's `full`
// barrier; the rest epilogue.  `full` thus completes when the code tiles
// have landed (the producer's byte count) and the scales are in TMEM (the
// copier's commit), and the MMA issuer waits once per K block.  Warps 0-2
// run their loops on all 32 lanes; one elected lane issues each copy, MMA
// and commit (issued from a one-lane branch instead, the same kernel took
// 167.6 µs on MXFP4 8192³ against 156.3 µs).  Copies issued
// from the MMA lane itself, just before the MMAs that read them, put each
// copy's latency in front of those MMAs (MXFP4 8192³: 180 -> 248 µs); from
// a separate warp they run ahead.  The scales
// travel in the compact chunk order (1 KB per 128 rows and K block) and are
// replicated across the TMEM lane quarters by the copies themselves
// (32x128b.warpx4): a quarter of the L2 traffic and of the relayout output
// of the 4x replicated form that three wide 128x256b copies would read
// (209 -> 197 µs).  TMEM per CTA: the accumulator(s) plus, per stage,
// 8 columns of A scales and 8·ceil(BN/128) columns of B scales (B rows 0-127
// in the first 4 columns of each K-block group, rows 128.. in the next 4).
// A stage's scale columns are rewritten only after its `sfull` barrier
// completes again, which needs the producer to have refilled the stage after
// its `empty` commit — issued after the MMAs that read those columns — so
// the copier never overwrites scales still in use.
//
// Every role waits on its own CTA's barriers with CTA-scope acquire: a wait
// at cluster scope cost the producer enough to slow the whole kernel (MXFP4
// 8192³: 180 -> 172 µs).  The epilogue stores D with 32-byte vector stores
// when rows allow it, so each store writes whole 32-byte sectors (172 ->
// 166 µs: half-sector stores doubled the write traffic into L2).
//
// The FlyDSL pages express the product with scaled MFMA/WMMA atoms (E8M0
// scale per 32 K elements: "FlyDSL Kernel Authoring Skill", §6, MX-scaled
// WMMA; "Kernel authoring guide", §4.3 GFX950 scaled MFMA).
#include <cuda_bf16.h>

#include <cstring>

#include "mx_common.cuh"

namespace tmg {
namespace {

using namespace mx;

constexpr int kBM = 256;
constexpr int kHalfM = 128;
// Scale form in shared memory: wide (each 512-byte chunk repeated four times,
// three tcgen05.cp 128x256b per K block) or compact (one copy of each chunk,
// 2 + 2·NSUB tcgen05.cp 32x128b.warpx4 that replicate across the lane
// quarters themselves).
constexpr bool kWideScales = false;
// warps 0-2 (producer, MMA, scale copier) + epilogue warps: 4 with two
// accumulators, 8 with one (two warps per TMEM lane quarter, each draining
// half the columns)
constexpr int kFirstEpiWarp = 3;
__host__ __device__ constexpr int pair_threads(int acc_bufs) { return acc_bufs == 1 ? 352 : 224; }
constexpr int kGroupM = 8;
constexpr int kTmemCols = 512;

template <int BN, int ACC_BUFS>
struct MxPairCfg {
    static constexpr int NSUB = (BN + 127) / 128;
    static constexpr int A_BYTES = kHalfM * kBKBytes;          // 16 KB
    static constexpr int B_BYTES = (BN / 2) * kBKBytes;
    static constexpr int SFA_BYTES = kWideScales ? kWideSrcBytes : kSfBlock;
    static constexpr int SFB_BYTES = NSUB * SFA_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int SF_COLS = 8 + 8 * NSUB;                 // per stage
    static constexpr int TMEM_STAGES = (kTmemCols - ACC_BUFS * BN) / SF_COLS;
    static constexpr int SMEM_STAGES = (230 * 1024 - 2048) / STAGE_BYTES;
    static constexpr int STAGES0 = TMEM_STAGES < SMEM_STAGES ? TMEM_STAGES : SMEM_STAGES;
    static constexpr int STAGES = STAGES0 > 8 ? 8 : STAGES0;
    static constexpr int CODE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SCALE_BYTES = SFA_BYTES + SFB_BYTES;
    static constexpr int BAR_BYTES = (3 * STAGES + 4) * 8 + 16;
    static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
};

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &tm, int &tn)
{
    const int group = kGroupM * tiles_n;
    const int first_m = (t / group) * kGroupM;
    const int gm = min(tiles_m - first_m, kGroupM);
    const int r = t % group;
    tm = first_m + r % gm;
    tn = r / gm;
}

// ACC_BUFS = 2: two accumulators, the epilogue of tile i overlaps the
// mainloop of tile i+1.  ACC_BUFS = 1 (BN = 256, where two accumulators
// would leave no TMEM for scales): the epilogue first drains the whole
// accumulator into packed bf16 registers, releases TMEM, then stores.
template <int BN, int ACC_BUFS>
__global__ void __launch_bounds__(pair_threads(ACC_BUFS), 1)
    mxfp4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                      __nv_bfloat16 *__restrict__ D, int M, int N, int K, int vec_ok, ErrCtx err)
{
    using C = MxPairCfg<BN, ACC_BUFS>;
    constexpr int STAGES = C::STAGES;
    constexpr int NSUB = C::NSUB;
    const int64_t d_limit = static_cast<int64_t>(M) * N;     // elements of D
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *tA = smem;
    uint8_t *tB = tA + STAGES * C::A_BYTES;
    uint8_t *sfA = tB + STAGES * C::B_BYTES;
    uint8_t *sfB = sfA + STAGES * C::SFA_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(sfB + STAGES * C::SFB_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *sfull = tempty + 2;                      // the stage's scales have landed in shared memory
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sfull + STAGES);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_kb = K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 2);      // the producer's byte count + the copier's commit
            mbar_init(&empty[s], 1);
            mbar_init(&sfull[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 2 * (pair_threads(ACC_BUFS) / 32 - kFirstEpiWarp));   // epilogue warps of both CTAs
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------- TMA producer
        // The kernel is a programmatic dependent launch of the scale
        // relayout pre-pass: the first ring's worth of code tiles is
        // requested before waiting for the pre-pass, their scale loads
        // right after it.
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        bool scales_ready = false;
        // rows (of 256 bytes) of this CTA's relaid scales for tile t, K block kb
        auto sfa_row = [&](int tm, int kb) {
            return (tm * 2 + static_cast<int>(rank)) * num_kb * (C::SFA_BYTES / 256) + kb * (C::SFA_BYTES / 256);
        };
        auto sfb_row = [&](int tn, int kb) { return tn * num_kb * (C::SFB_BYTES / 256) + kb * (C::SFB_BYTES / 256); };
        auto load_scales = [&](int st, int tm, int tn, int kb) {
            const uint32_t b0 = mapa_shared(smem_u32(&sfull[st]), 0);
            tma_load_2d_pair_w(sfA + st * C::SFA_BYTES, &tmSA, b0, 0, sfa_row(tm, kb));
            tma_load_2d_pair_w(sfB + st * C::SFB_BYTES, &tmSB, b0, 0, sfb_row(tn, kb));
        };
        // the units issued so far are the first ones of this pair's walk,
        // in stages 0, 1, ...: load their scales
        auto release_deferred = [&]() {
            griddep_wait();
            int64_t i = 0;
            for (int t2 = cluster; t2 < num_tiles && i < issued; t2 += nclusters) {
                int tm2, tn2;
                tile_coords(t2, tiles_m, tiles_n, tm2, tn2);
                for (int kb2 = 0; kb2 < num_kb && i < issued; ++kb2, ++i)
                    load_scales(static_cast<int>(i), tm2, tn2, kb2);
            }
            scales_ready = true;
        };
        for (int t = cluster; t < num_tiles && ok; t += nclusters) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!scales_ready && issued == STAGES)
                    release_deferred();
                if (!mbar_wait_warp(&empty[stage], phase ^ 1u, err, abort_flag, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                if (rank == 0) {
                    // codes and scales complete on separate barriers, so
                    // that the scale copies need not wait for the codes
                    mbar_arrive_expect_tx_w(&full[stage], 2 * C::CODE_BYTES);
                    mbar_arrive_expect_tx_w(&sfull[stage], 2 * C::SCALE_BYTES);
                }
                const uint32_t bar0 = mapa_shared(smem_u32(&full[stage]), 0);
                tma_load_2d_pair_w(tA + stage * C::A_BYTES, &tmA, bar0, kb * kBKBytes,
                                   tm * kBM + static_cast<int>(rank) * kHalfM);
                tma_load_2d_pair_w(tB + stage * C::B_BYTES, &tmB, bar0, kb * kBKBytes,
                                   tn * BN + static_cast<int>(rank) * (BN / 2));
                if (scales_ready)
                    load_scales(stage, tm, tn, kb);
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!scales_ready)
            release_deferred();          // fewer units than stages, or an early stop
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
            // (warp 1 and warp 2 each run their loop on the whole warp; one
            // elected lane issues)
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters, ++local) {
                const int acc = local % ACC_BUFS;
                const uint32_t use_phase = (local / ACC_BUFS) & 1;
                if (!mbar_wait_warp(&tempty[acc], use_phase ^ 1u, err, abort_flag, kSiteMmaTmemEmpty))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    // the stage's codes are in shared memory, its scales in TMEM
                    if (!mbar_wait_warp(&full[stage], phase, err, abort_flag, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_col = tmem_base + ACC_BUFS * BN + stage * C::SF_COLS;
                    const uint32_t sfb_col = sfa_col + 8;
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(tA + stage * C::A_BYTES));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(tB + stage * C::B_BYTES));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t koff = static_cast<uint64_t>((k * 32) >> 4);
                        const int c = k >> 1;
                        const uint32_t id = (k & 1) ? 2u : 0u;
                        mma_mxf4_pair_w(d_tmem, adesc + koff, bdesc + koff, idesc_mxf4(kBM, BN, id), sfa_col + c * 4,
                                      sfb_col + c * 4 * NSUB, (kb | k) != 0);
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
    } else if (warp == 2) {
        if (rank == 0) {
            // --------------------------------------------- scale copier
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters) {
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_warp(&sfull[stage], phase, err, abort_flag, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_col = tmem_base + ACC_BUFS * BN + stage * C::SF_COLS;
                    const uint32_t sfb_col = sfa_col + 8;
                    // 1 + NSUB wide copies: A scales (both K-block groups),
                    // then B scales per K-block group (NSUB = 2) or both
                    // groups at once (NSUB = 1)
                    if constexpr (kWideScales) {
                        tmem_cp_wide_pair_w(sfa_col, sdesc_wide_scales(smem_u32(sfA + stage * C::SFA_BYTES)));
#pragma unroll
                        for (int p = 0; p < NSUB; ++p)
                            tmem_cp_wide_pair_w(sfb_col + 8 * p,
                                              sdesc_wide_scales(smem_u32(sfB + stage * C::SFB_BYTES + p * kWideSrcBytes)));
                    } else {
                        // chunk c (scale blocks 4c..4c+3) of sub-block s
                        // -> columns c * 4 * NSUB + 4 s of the group
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            tmem_cp_chunk_pair_w(sfa_col + 4 * c,
                                               sdesc_noswizzle_rows16(smem_u32(sfA + stage * C::SFA_BYTES + c * kSfChunk)));
#pragma unroll
                            for (int sb = 0; sb < NSUB; ++sb)
                                tmem_cp_chunk_pair_w(sfb_col + c * 4 * NSUB + 4 * sb,
                                                   sdesc_noswizzle_rows16(smem_u32(sfB + stage * C::SFB_BYTES +
                                                                                   sb * kSfBlock + c * kSfChunk)));
                        }
                    }
                    mma_commit_pair_w(&full[stage], 0x1);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;
        int local = 0;
        for (int t = cluster; t < num_tiles; t += nclusters, ++local) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            const int acc = local % ACC_BUFS;
            if (!mbar_wait_cluster(&tfull[acc], (local / ACC_BUFS) & 1, err, abort_flag, kSiteEpiTmemFull))
                break;
            tc_fence_after();
            const int row = tm * kBM + static_cast<int>(rank) * kHalfM + q * 32 + lane;
            __nv_bfloat16 *drow = D + static_cast<int64_t>(row) * N;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            if constexpr (ACC_BUFS == 1) {
                // drain this warp's half of the columns first so the next
                // tile's MMAs can start, then store
                constexpr int HALF = BN / 2;
                const int h = (warp - kFirstEpiWarp) / 4;
                uint32_t packed[HALF / 2];
#pragma unroll
                for (int c = 0; c < HALF / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tbase + h * HALF + c * 32, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        packed[c * 16 + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
                if (row < M) {
#pragma unroll
                    for (int c = 0; c < HALF / 32; ++c) {
                        const int col0 = tn * BN + h * HALF + c * 32;
                        if (col0 >= N || !span_ok(static_cast<int64_t>(row) * N + col0, min(32, N - col0), d_limit, err,
                                                  kBndStoreD))
                            continue;
                        if (vec_ok == 2 && col0 + 32 <= N) {
                            const uint32_t *w = packed + c * 16;
                            st_global_v8(drow + col0, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                            st_global_v8(drow + col0 + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
                        } else if (vec_ok && col0 + 32 <= N) {
                            uint4 *dst = reinterpret_cast<uint4 *>(drow + col0);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                dst[j] = make_uint4(packed[c * 16 + 4 * j], packed[c * 16 + 4 * j + 1],
                                                    packed[c * 16 + 4 * j + 2], packed[c * 16 + 4 * j + 3]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (col0 + j < N) {
                                    const uint32_t w = packed[c * 16 + j / 2];
                                    const uint16_t hv = (j & 1) ? static_cast<uint16_t>(w >> 16)
                                                                : static_cast<uint16_t>(w & 0xFFFFu);
                                    drow[col0 + j] = __ushort_as_bfloat16(hv);
                                }
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tbase + c * 32, v);
                    const int col0 = tn * BN + c * 32;
                    if (row < M && col0 < N &&
                        span_ok(static_cast<int64_t>(row) * N + col0, min(32, N - col0), d_limit, err, kBndStoreD)) {
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
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <int BN, int ACC_BUFS>
cudaError_t launch_pair(const Mxfp4Args &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    using C = MxPairCfg<BN, ACC_BUFS>;
    static_assert(C::STAGES >= 3, "pipeline depth");
    static_assert(C::SMEM <= 232448, "shared memory budget");
    static_assert(ACC_BUFS * BN + C::STAGES * C::SF_COLS <= kTmemCols, "TMEM budget");
    static_assert(C::B_BYTES % 1024 == 0, "B half must be whole 8-row swizzle atoms");
    auto kern = mxfp4_pair_kernel<BN, ACC_BUFS>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM);
    if (e != cudaSuccess)
        return e;
    e = launch_mx_scale_relayout(a.sA, a.M, a.relA, kHalfM, a.sB, a.N, a.relB, BN, a.K, kWideScales, num_sms, s);
    if (e != cudaSuccess)
        return e;
    const int tiles = ((a.M + kBM - 1) / kBM) * ((a.N + BN - 1) / BN);
    int clusters = num_sms / 2;
    if (tiles < clusters)
        clusters = tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(pair_threads(ACC_BUFS));
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlaps the relayout pre-pass
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // row stores: 2 = 32-byte vectors (rows start on 32-byte boundaries), 1 = 16-byte vectors, 0 = scalars
    const uintptr_t d_addr = reinterpret_cast<uintptr_t>(a.D);
    const int vec_ok = (a.N % 16 == 0 && (d_addr & 31u) == 0) ? 2 : (a.N % 8 == 0 && (d_addr & 15u) == 0) ? 1 : 0;
    note_launch();
    e = cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.tmSA, a.tmSB, static_cast<__nv_bfloat16 *>(a.D), a.M, a.N,
                           a.K, vec_ok, err);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace

bool mxfp4_pair_wide_scales() { return kWideScales; }

int mxfp4_pair_pick_bn(int64_t M, int64_t N, int num_sms)
{
    static const int cands[] = {256, 192, 128};
    const int64_t clusters = num_sms / 2;
    const int64_t tm = (M + kBM - 1) / kBM;
    int best = 256;
    int64_t best_cost = -1;
    for (int bn : cands) {
        const int64_t tiles = tm * ((N + bn - 1) / bn);
        const int64_t cost = ((tiles + clusters - 1) / clusters) * (bn + 48);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

cudaError_t launch_mxfp4_pair(const Mxfp4Args &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    if (a.bn == 256)
        return launch_pair<256, 1>(a, num_sms, err, s);
    if (a.bn == 192)
        return launch_pair<192, 2>(a, num_sms, err, s);
    return launch_pair<128, 2>(a, num_sms, err, s);
}

}  // namespace tmg
