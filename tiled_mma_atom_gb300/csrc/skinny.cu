// skinny.cu — decode-shaped GEMM (M <= 64, N and K large) on tcgen05 with
// the operands swapped: Dᵀ (N x M) = B (N x K) · A (M x K)ᵀ.  The 128-row MMA
// dimension runs over N (rows of B, the weight matrix streamed from HBM) and
// the small M becomes the MMA's N (16..64), so no tensor-core lane idles on
// padding rows.  The work is HBM-bound: the point is to keep enough TMA
// loads of B in flight on every SM.
//
// The pages' preshuffle GEMM takes a runtime M so one kernel serves any
// batch ("Kernel authoring guide", §11, note under the example); the skinny
// case is the small-M end of that range.
//
// Work split: the units are (128-row tile of B, 64-wide K block).  Each of
// the G CTAs takes tiles / G whole tiles (data-parallel, written directly)
// and an equal contiguous run of the units of the remaining tiles mod G
// (stream-K), which it runs first.  Partial tiles write fp32 partial sums
// to scratch; the last CTA to arrive at a tile (a counter per tile and TMEM
// lane quarter, so each epilogue warp settles its own 32 rows) adds all
// partials in CTA order — a fixed order, so results do not depend on
// timing — rounds to bf16, writes D, and resets the counter to zero for the
// next call.  With the split tiles first, those fix-ups overlap the
// streaming of the whole tiles.  At 16 x 28672 x 8192 (224 tiles on 152
// CTAs: one whole tile each plus 72 tiles shared out) the call takes 76.4
// us against 78.5 us when every CTA's run ended on a split tile.
//
// Roles as in tc_bf16.cu: warp 0 TMA producer, warp 1 MMA issuer (and TMEM
// owner), warps 2..5 epilogue; 8-stage ring of 16 KB (B) + mp·128 B (A).
#include <cuda_bf16.h>

#include <map>
#include <mutex>

#include "internal.h"

namespace tmg {
namespace {

constexpr int kTileN = 128;        // rows of B per tile (MMA M)
constexpr int kBK = 64;
constexpr int kUmmaK = 16;
constexpr int kStages = 8;
constexpr int kMaxMP = 64;
constexpr int kBBytes = kTileN * kBK * 2;        // 16 KB
constexpr int kABytesMax = kMaxMP * kBK * 2;     // 8 KB
constexpr int kStageBytes = kBBytes + kABytesMax;
constexpr int kTmemCols = 2 * kMaxMP;            // 128
constexpr int kSmem = kStages * kStageBytes + (2 * kStages + 4) * 8 + 32 + 1024;
constexpr int kThreads = 192;

__device__ __forceinline__ int64_t unit_start(int c, int64_t U, int G)
{
    return (static_cast<int64_t>(c) * U) / G;
}

// The work of CTA c of G: first its stream-K run [b, e) over the units of
// the first sk_tiles tiles (split at tile boundaries into segments), then its
// data-parallel tiles sk_tiles + c + j G, j < dpc, each whole.  With dpc =
// tiles / G whole tiles per CTA and the remaining sk_tiles = tiles mod G
// shared out as equal runs of units, every CTA streams the same number of
// bytes, and the split tiles (whose partial sums the last contributing CTA
// adds up) come first: their fix-ups overlap the whole tiles' streaming,
// and every CTA ends on a whole tile, written directly.
struct Work {
    int64_t b, e;
    int KB, t0, nsk, dpc, sk_tiles, c, G;
    __device__ Work(int c_, int G_, int tiles, int kb) : KB(kb), c(c_), G(G_)
    {
        dpc = tiles / G;
        sk_tiles = tiles - dpc * G;
        // every CTA needs at least one stream-K unit (the fix-up counts on
        // each CTA between a split tile's first and last owners): with
        // fewer units than CTAs, one more wave of tiles joins the stream-K
        // region
        if (sk_tiles > 0 && static_cast<int64_t>(sk_tiles) * KB < G && dpc > 0) {
            --dpc;
            sk_tiles += G;
        }
        const int64_t U = static_cast<int64_t>(sk_tiles) * KB;
        b = unit_start(c, U, G);
        e = unit_start(c + 1, U, G);
        t0 = static_cast<int>(b / KB);
        nsk = b < e ? static_cast<int>((e - 1) / KB) - t0 + 1 : 0;
    }
    __device__ int count() const { return nsk + dpc; }
    // tile and K-block range [kb0, kb1) of the p-th segment
    __device__ void get(int p, int &tile, int &kb0, int &kb1) const
    {
        if (p < nsk) {
            const int64_t u0 = p == 0 ? b : static_cast<int64_t>(t0 + p) * KB;
            const int64_t end = static_cast<int64_t>(t0 + p + 1) * KB;
            const int64_t u1 = end < e ? end : e;
            tile = static_cast<int>(u0 / KB);
            kb0 = static_cast<int>(u0 % KB);
            kb1 = kb0 + static_cast<int>(u1 - u0);
        } else {
            tile = sk_tiles + c + (p - nsk) * G;
            kb0 = 0;
            kb1 = KB;
        }
    }
};

// CTA whose run contains unit u.
__device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int G)
{
    return static_cast<int>(((u + 1) * G - 1) / U);
}

__global__ void __launch_bounds__(kThreads, 1)
    skinny_tc_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA,
                     __nv_bfloat16 *__restrict__ D, int64_t ldd, int M, int N, int K, int mp,
                     float *__restrict__ partials, uint32_t *__restrict__ counters, ErrCtx err)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int G = gridDim.x, c = blockIdx.x;
    const int tiles = (N + kTileN - 1) / kTileN;
    const int KB = (K + kBK - 1) / kBK;
    const Work work(c, G, tiles, KB);
    const int64_t U = static_cast<int64_t>(work.sk_tiles) * KB;      // stream-K units
    const int64_t d_limit = static_cast<int64_t>(M - 1) * ldd + N;                   // elements of D
    const int64_t p_limit = static_cast<int64_t>(G) * 2 * mp * kTileN;               // floats of partials
    const uint32_t a_bytes = static_cast<uint32_t>(mp) * kBK * 2;

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
        const uint64_t keep_a = policy_evict_last();   // A is re-read by every CTA
        const uint64_t stream_b = policy_evict_first(); // B is read once
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        for (int p = 0; p < work.count() && ok; ++p) {
            int tile, kb0, kb1;
            work.get(p, tile, kb0, kb1);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_warp(&empty[stage], phase ^ 1u, err, abort_flag, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + stage * kStageBytes;
                mbar_arrive_expect_tx_w(&full[stage], kBBytes + a_bytes);
                tma_load_2d_hint_w(st, &tmB, &full[stage], kb * kBK, tile * kTileN, stream_b);
                tma_load_2d_hint_w(st + kBBytes, &tmA, &full[stage], kb * kBK, 0, keep_a);
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
        // (the whole warp runs the issue loop; one elected lane issues)
        const uint32_t idesc = idesc_bf16_f32(kTileN, mp);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int seg = 0; seg < work.count() && ok; ++seg) {
            int tile, kb0, kb1;
            work.get(seg, tile, kb0, kb1);
            const int acc = seg & 1;
            if (!mbar_wait_warp(&tempty[acc], ((seg >> 1) & 1) ^ 1u, err, abort_flag, kSiteMmaTmemEmpty))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * kMaxMP;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_warp(&full[stage], phase, err, abort_flag, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint8_t *st = smem + stage * kStageBytes;
                const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(st));            // MMA "A": B rows
                const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(st + kBBytes));  // MMA "B": A rows
#pragma unroll
                for (int k = 0; k < kBK / kUmmaK; ++k) {
                    const uint64_t koff = static_cast<uint64_t>((k * kUmmaK * 2) >> 4);
                    mma_bf16_w(d_tmem, bdesc + koff, adesc + koff, idesc, (kb != kb0) || (k != 0));
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
        // epilogue: thread owns B row n_local = 32 q + lane of the tile
        const int q = warp & 3;
        const int n_local = q * 32 + lane;
        for (int seg = 0; seg < work.count(); ++seg) {
            int tile, kb0, kb1;
            work.get(seg, tile, kb0, kb1);
            const int acc = seg & 1;
            if (!mbar_wait(&tfull[acc], (seg >> 1) & 1, err, abort_flag, kSiteEpiTmemFull))
                break;
            tc_fence_after();
            float v[kMaxMP];
#pragma unroll
            for (int ch = 0; ch < kMaxMP / 16; ++ch) {
                if (ch * 16 < mp) {
                    uint32_t r[16];
                    tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kMaxMP + ch * 16, r);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[ch * 16 + j] = __uint_as_float(r[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[ch * 16 + j] = 0.f;
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
                        if (m < M && bounds_ok(static_cast<int64_t>(m) * ldd + n, d_limit, err, kBndStoreD))
                            D[static_cast<int64_t>(m) * ldd + n] = __float2bfloat16_rn(v[m]);
                }
                continue;
            }
            // Partial tile: publish this warp's 32 rows; the last warp to
            // arrive for (tile, quarter) reduces them.  Warps never wait on
            // one another, so an aborted warp cannot stall the others.
            const int slot = 2 * c + (tile == work.t0 ? 0 : 1);
            const int64_t mine_off = static_cast<int64_t>(slot) * mp * kTileN;
            float *mine = partials + mine_off;
#pragma unroll
            for (int m = 0; m < kMaxMP; ++m)
                if (m < mp && bounds_ok(mine_off + m * kTileN + n_local, p_limit, err, kBndPartials))
                    mine[m * kTileN + n_local] = v[m];
            __threadfence();
            __syncwarp();
            const int64_t t_first = static_cast<int64_t>(tile) * KB;
            const int c_first = unit_owner(t_first, U, G);
            const int c_last = unit_owner(t_first + KB - 1, U, G);
            if (!bounds_ok(static_cast<int64_t>(tile) * 4 + q, static_cast<int64_t>(tiles) * 4, err, kBndCounters))
                continue;
            uint32_t old = 0;
            if (lane == 0)
                old = atomicAdd(&counters[tile * 4 + q], 1u);
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == static_cast<uint32_t>(c_last - c_first)) {
                __threadfence();
                float sum[kMaxMP];
#pragma unroll
                for (int m = 0; m < kMaxMP; ++m)
                    sum[m] = 0.f;
                for (int cc = c_first; cc <= c_last; ++cc) {
                    if (cc == c) {
#pragma unroll
                        for (int m = 0; m < kMaxMP; ++m)
                            sum[m] += v[m];
                    } else {
                        const int first_tile = static_cast<int>(unit_start(cc, U, G) / KB);
                        const int s2 = 2 * cc + (first_tile == tile ? 0 : 1);
                        const int64_t p_off = static_cast<int64_t>(s2) * mp * kTileN;
                        const float *p = partials + p_off;
#pragma unroll
                        for (int m = 0; m < kMaxMP; ++m)
                            if (m < mp && bounds_ok(p_off + m * kTileN + n_local, p_limit, err, kBndPartials))
                                sum[m] += __ldcg(p + m * kTileN + n_local);
                    }
                }
                if (n < N) {
#pragma unroll
                    for (int m = 0; m < kMaxMP; ++m)
                        if (m < M && bounds_ok(static_cast<int64_t>(m) * ldd + n, d_limit, err, kBndStoreD))
                            D[static_cast<int64_t>(m) * ldd + n] = __float2bfloat16_rn(sum[m]);
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

size_t skinny_partials_bytes(int grid, int mp)
{
    return static_cast<size_t>(grid) * 2 * mp * kTileN * sizeof(float);
}

size_t skinny_counters_bytes(int64_t N)
{
    return static_cast<size_t>((N + kTileN - 1) / kTileN) * 4 * sizeof(uint32_t);
}

cudaError_t launch_skinny_tc(const SkinnyTcArgs &a, const ErrCtx &err, cudaStream_t s)
{
    static_assert(kSmem <= 232448, "shared memory budget");
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(skinny_tc_kernel), kSmem);
    if (e != cudaSuccess)
        return e;
    note_launch();
    skinny_tc_kernel<<<a.grid, kThreads, kSmem, s>>>(a.tmB, a.tmA, static_cast<__nv_bfloat16 *>(a.D), a.ldd,
                                                     a.M, a.N, a.K, a.mp, a.partials, a.counters, err);
    return cudaGetLastError();
}

}  // namespace tmg

namespace tmg {

// ---------------------------------------------------------------------------
// Fixed-scratch variant.
//
// Some callers cannot allocate device memory when they call the GEMM: for
// example a latency-critical loop that must not call cudaMalloc/cudaFree
// after start-up (both can synchronise the whole device), or a plug-in whose
// host application owns all device memory through its own pool and gives
// the plug-in only the input and output buffers.  For them the skinny kernel
// can take its split-K partial sums and per-tile counters from one array in
// static device memory instead of from scratch that the ordinary call
// allocates per stream.  The array is part of the library's device image:
// every GPU that loads the library holds it until the process exits.
namespace {

constexpr size_t kFixedScratchBytes = size_t(8) << 20;                      // 8 MiB
constexpr int kFixedMaxTiles = 4096;                                          // N <= 524288
constexpr size_t kFixedCounterBytes = size_t(kFixedMaxTiles) * 4 * sizeof(uint32_t);  // 64 KiB

static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

std::mutex g_fixed_mu;
std::map<int, unsigned char *> g_fixed_addr;    // device ordinal -> device address

}  // namespace

cudaError_t skinny_fixed_scratch(FixedScratch *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_fixed_mu);
    auto it = g_fixed_addr.find(dev);
    if (it == g_fixed_addr.end()) {
        // In host code `g_fixed_scratch` names a host-side stand-in, not device
        // memory: the kernel must get the address the runtime reports for the
        // current device.
        unsigned char *p = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_fixed_scratch);
        if (e != cudaSuccess)
            return e;
        it = g_fixed_addr.emplace(dev, p).first;
    }
    out->counters = reinterpret_cast<uint32_t *>(it->second);
    out->counter_bytes = kFixedCounterBytes;
    out->partials = reinterpret_cast<float *>(it->second + kFixedCounterBytes);
    out->partial_bytes = kFixedScratchBytes - kFixedCounterBytes;
    out->max_tiles = kFixedMaxTiles;
    return cudaSuccess;
}

}  // namespace tmg
