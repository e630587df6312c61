// tc2_bf16.cu — the bf16 GEMM of tc_bf16.cu on CTA pairs: each cluster of
// two CTAs computes a 256 x BN output tile with tcgen05.mma.cta_group::2
// (M = 256).  CTA r (r = 0, 1) holds rows 128r..128r+127 of the A tile and
// rows r·BN/2 .. (r+1)·BN/2 - 1 of the B tile in its own shared memory, so
// each SM loads half the B tile it would need alone: per SM and K block,
// 16 KB of A plus BN/2 x 128 bytes of B instead of 16 KB plus BN x 128 bytes.
//
// Roles, in both CTAs unless stated:
//   warp 0        TMA producer for this CTA's halves; the loads of both CTAs
//                 complete on CTA 0's `full` barrier (CTA 0 announces the
//                 pair's byte count); waits on its own `empty` barrier.
//   warp 1        CTA 0 only: issues the pair MMAs and commits with a
//                 multicast arrive on the `empty` / `tmem_full` barriers of
//                 both CTAs.  Both CTAs' warp 1 allocate TMEM together.
//   warps 2..5    epilogue of this CTA's 128 accumulator rows; each warp
//                 then arrives on CTA 0's `tmem_empty` barrier (count 8).
// Tile widths 128..256: the host picks the one that best fills the last wave
// (e.g. 224 for 4096 x 4096: 16 x 19 tiles = exactly 4 waves of 76 pairs).
#include <cuda_bf16.h>

#include <cstring>

#include "internal.h"

namespace tmg {
namespace {

constexpr int kBM = 256;           // rows per pair tile
constexpr int kHalfM = 128;        // rows per CTA
constexpr int kBK = 64;
constexpr int kUmmaK = 16;
constexpr int kThreads = 192;
constexpr int kGroupM = 8;

template <int BN>
struct PairCfg {
    static constexpr int A_BYTES = kHalfM * kBK * 2;            // 16 KB
    static constexpr int B_BYTES = (BN / 2) * kBK * 2;          // this CTA's half
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (220 * 1024 - 2048) / STAGE_BYTES > 8 ? 8 : (220 * 1024 - 2048) / STAGE_BYTES;
    static constexpr int TMEM_COLS = 512;
    static constexpr int BAR_BYTES = (2 * STAGES + 4) * 8 + 16;
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

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tc2_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    __nv_bfloat16 *__restrict__ D, int64_t ldd, int M, int N, int K, int vec_ok,
                    ErrCtx err)
{
    using C = PairCfg<BN>;
    constexpr int STAGES = C::STAGES;
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

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_kb = (K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);
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
        if (lane == 0) {
            // ---------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters) {
                int tm, tn;
                tile_coords(t, tiles_m, tiles_n, tm, tn);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_cluster(&empty[stage], phase ^ 1u, err, abort_flag, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0)
                        mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                    const uint32_t bar0 = mapa_shared(smem_u32(&full[stage]), 0);
                    tma_load_2d_pair(sA + stage * C::A_BYTES, &tmA, bar0, kb * kBK, tm * kBM + rank * kHalfM);
                    tma_load_2d_pair(sB + stage * C::B_BYTES, &tmB, bar0, kb * kBK, tn * BN + rank * (BN / 2));
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
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, err, abort_flag, kSiteMmaTmemEmpty))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_cluster(&full[stage], phase, err, abort_flag, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + stage * C::A_BYTES));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        const uint64_t koff = static_cast<uint64_t>((k * kUmmaK * 2) >> 4);
                        mma_bf16_pair(d_tmem, adesc + koff, bdesc + koff, idesc, (kb | k) != 0);
                    }
                    mma_commit_pair(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit_pair(&tfull[acc], 0x3);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;
        int local = 0;
        for (int t = cluster; t < num_tiles; t += nclusters, ++local) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait_cluster(&tfull[acc], acc_phase, err, abort_flag, kSiteEpiTmemFull))
                break;
            tc_fence_after();
            const int row = tm * kBM + static_cast<int>(rank) * kHalfM + q * 32 + lane;
            __nv_bfloat16 *drow = D + static_cast<int64_t>(row) * ldd;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * 32, v);
                const int col0 = tn * BN + c * 32;
                if (row < M) {
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

    __syncwarp();
    tc_fence_before();
    cluster_sync();          // no CTA leaves while its peer may still touch it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

template <int BN>
cudaError_t launch_pair(const TcArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    using C = PairCfg<BN>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    static_assert(2 * BN <= C::TMEM_COLS, "TMEM budget");
    static_assert(C::B_BYTES % 1024 == 0, "B half must be whole 8-row swizzle atoms");
    auto kern = tc2_bf16_kernel<BN>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM);
    if (e != cudaSuccess)
        return e;
    const int tiles = ((a.M + kBM - 1) / kBM) * ((a.N + BN - 1) / BN);
    int clusters = num_sms / 2;
    if (tiles < clusters)
        clusters = tiles;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
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
                           vec_ok, err);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace

int tc2_pick_bn(int64_t M, int64_t N, int num_sms)
{
    static const int cands[] = {256, 224, 192, 128};
    const int64_t clusters = num_sms / 2;
    const int64_t tm = (M + kBM - 1) / kBM;
    int best = 256;
    int64_t best_cost = -1;
    for (int bn : cands) {
        const int64_t tiles = tm * ((N + bn - 1) / bn);
        const int64_t waves = (tiles + clusters - 1) / clusters;
        // makespan in columns of work; +48 charges narrower tiles for their
        // higher operand traffic per flop and fixed per-tile cost
        const int64_t cost = waves * (bn + 48);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

cudaError_t launch_tc2_bf16(const TcArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    switch (a.bn) {
    case 256:
        return launch_pair<256>(a, num_sms, err, s);
    case 224:
        return launch_pair<224>(a, num_sms, err, s);
    case 192:
        return launch_pair<192>(a, num_sms, err, s);
    default:
        return launch_pair<128>(a, num_sms, err, s);
    }
}

}  // namespace tmg
