// tc_bf16.cu — persistent, warp-specialised tcgen05 GEMM for bf16:
// D (bf16, M x N) = A (M x K, K-major) · B (N x K, K-major)ᵀ, fp32 accumulate
// in tensor memory.
//
// The FlyDSL pages build the same operation for MI300X/MI350 as the
// preshuffle GEMM ("FlyDSL Kernel Authoring Skill", §6 "GEMM Pattern
// (Preshuffle)"; "Kernel authoring guide", §11 "Complete example"): A tiles
// staged in LDS with an XOR swizzle, two LDS stages so loads of step k+1
// overlap the MFMAs of step k (§3 "Runtime Loops with Loop-Carried Values"),
// and a direct row-major or LDS-shuffled epilogue.  On sm_103a the same roles
// map onto dedicated hardware:
//   warp 0        TMA producer: one elected lane issues cp.async.bulk.tensor
//                 tile loads (128-byte swizzle, out-of-range rows/columns
//                 read as zero) into a STAGES-deep shared-memory ring;
//                 mbarriers `full`/`empty` gate each stage.
//   warp 1        MMA issuer: one elected lane issues tcgen05.mma
//                 (kind::f16, 128 x BN x 16) from shared-memory descriptors
//                 into a TMEM
//                 accumulator; tcgen05.commit releases each stage and, at
//                 tile end, hands the accumulator to the epilogue.  Warp 1 also
//                 allocates and frees TMEM.
//   warps 2..5    epilogue: tcgen05.ld TMEM -> registers (warp w reads TMEM
//                 lanes 32(w%4)..32(w%4)+31 = tile rows), fp32 -> bf16 round to
//                 nearest even, 16-byte stores.
// Warps 0 and 1 run their loops on all 32 lanes in warp-uniform control flow;
// each TMA copy, tcgen05.mma and commit carries an elect.sync predicate.
// Two TMEM accumulators (2 x BN columns) let the epilogue of tile i overlap
// the mainloop of tile i+1.  The grid is one CTA per SM; CTA c takes tiles
// c, c + grid, ... in a grouped order (8 M-tiles per group) so concurrently
// running CTAs share A and B tiles in L2.
#include <cuda_bf16.h>

#include "internal.h"

namespace tmg {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;            // 64 bf16 = 128 bytes = one swizzle row
constexpr int kUmmaK = 16;
constexpr int kThreads = 192;
constexpr int kGroupM = 8;

template <int BN, int STAGES>
struct Cfg {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
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

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   __nv_bfloat16 *__restrict__ D, int64_t ldd, int M, int N, int K, int vec_ok,
                   ErrCtx err)
{
    const int64_t d_limit = static_cast<int64_t>(M - 1) * ldd + N;     // elements of D
    using C = Cfg<BN, STAGES>;
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
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------- TMA producer
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait_warp(&empty[stage], phase ^ 1u, err, abort_flag, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_w(&full[stage], C::STAGE_BYTES);
                tma_load_2d_w(sA + stage * C::A_BYTES, &tmA, &full[stage], kb * kBK, tm * kBM);
                tma_load_2d_w(sB + stage * C::B_BYTES, &tmB, &full[stage], kb * kBK, tn * BN);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Drain: every load issued must have landed before the CTA may
        // exit.  On the normal path the MMA warp consumed them all and
        // these waits return at once.
        for (int i = 0; i < STAGES; ++i) {
            // the stage before `stage` in ring order, walking backwards
            int s = stage - 1 - i;
            uint32_t ph = phase;
            if (s < 0) {
                s += STAGES;
                ph ^= 1u;
            }
            // only stages that were ever filled
            const int64_t issued = static_cast<int64_t>(num_kb) *
                                   ((num_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                    static_cast<int>(gridDim.x));
            if (i >= issued)
                break;
            mbar_wait(&full[s], ph, err, nullptr, kSiteDrain);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        // (the whole warp runs the loop; one elected lane issues)
        constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait_warp(&tempty[acc], acc_phase ^ 1u, err, abort_flag, kSiteMmaTmemEmpty))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait_warp(&full[stage], phase, err, abort_flag, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + stage * C::A_BYTES));
                const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                for (int k = 0; k < kBK / kUmmaK; ++k) {
                    // advance 32 bytes (16 bf16) along K inside the swizzle row
                    const uint64_t koff = static_cast<uint64_t>((k * kUmmaK * 2) >> 4);
                    mma_bf16_w(d_tmem, adesc + koff, bdesc + koff, idesc, (kb | k) != 0);
                }
                mma_commit_w(&empty[stage]);
                if (++stage == STAGES) {
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
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        int local = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait(&tfull[acc], acc_phase, err, abort_flag, kSiteEpiTmemFull))
                break;
            tc_fence_after();
            const int row = tm * kBM + q * 32 + lane;
            __nv_bfloat16 *drow = D + static_cast<int64_t>(row) * ldd;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * 32, v);
                const int col0 = tn * BN + c * 32;
                const int64_t off = static_cast<int64_t>(row) * ldd + col0;
                if (row < M) {
                    if (vec_ok && col0 + 32 <= N) {
                        if (!span_ok(off, 32, d_limit, err, kBndStoreD))
                            continue;
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
                            if (col0 + j < N && bounds_ok(off + j, d_limit, err, kBndStoreD))
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
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int STAGES>
cudaError_t launch_cfg(const TcArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    using C = Cfg<BN, STAGES>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    auto kern = tc_bf16_kernel<BN, STAGES>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM);
    if (e != cudaSuccess)
        return e;
    const int tiles = ((a.M + kBM - 1) / kBM) * ((a.N + BN - 1) / BN);
    const int grid = tiles < num_sms ? tiles : num_sms;
    const int vec_ok = (a.ldd % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.D) & 15u) == 0);
    note_launch();
    kern<<<grid, kThreads, C::SMEM, s>>>(a.tmA, a.tmB, static_cast<__nv_bfloat16 *>(a.D), a.ldd,
                                         a.M, a.N, a.K, vec_ok, err);
    return cudaGetLastError();
}

}  // namespace

int tc_pick_bn(int64_t M, int64_t N, int64_t K, int num_sms, double *est_ns)
{
    // Per K block of one 128 x bn tile, measured on GB300 (bf16, L2 flushed,
    // M, N 1024-3072, K 1024-4096): 173 / 223 / 367 ns at widths 64 / 128 /
    // 256; whole waves of num_sms tiles.
    static const int widths[3] = {64, 128, 256};
    static const double cost[3] = {173.0, 223.0, 367.0};
    const int64_t num_kb = (K + kBK - 1) / kBK;
    const int64_t rows = (M + kBM - 1) / kBM;
    int best = 128;
    double best_t = -1.0;
    for (int i = 0; i < 3; ++i) {
        const int64_t tiles = rows * ((N + widths[i] - 1) / widths[i]);
        const double t = static_cast<double>((tiles + num_sms - 1) / num_sms) * num_kb * cost[i];
        if (best_t < 0.0 || t < best_t) {
            best_t = t;
            best = widths[i];
        }
    }
    if (est_ns)
        *est_ns = best_t;
    return best;
}

cudaError_t launch_tc_bf16(const TcArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    if (a.bn == 256)
        return launch_cfg<256, 4>(a, num_sms, err, s);
    if (a.bn == 64)
        return launch_cfg<64, 8>(a, num_sms, err, s);
    return launch_cfg<128, 6>(a, num_sms, err, s);
}

}  // namespace tmg
