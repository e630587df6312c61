// w4a8_skinny.cu — decode-shaped W4A8 GEMM (M <= 64): int8 activations A
// (M, K) x packed int4 weights B (N, K/2) -> exact int32 D (M, N), reading
// only the 4-bit weights from HBM.
//
// The pages' W4A8 kernel unpacks the int4 B to int8 in the kernel and uses
// an i8 x i8 -> i32 atom ("FlyDSL Kernel Authoring Skill", §10 item 10; §6
// integer WMMA rows).  GB300 has no integer tensor-core MMA, so the product
// runs as tcgen05 kind::f8f6f4 (E4M3 operands, fp32 accumulation) on values
// that E4M3 holds exactly:
//   * weights in offset binary: u = v + 8 = nibble XOR 8, in 0..15.  The
//     E4M3 codes 0..15 (exponent field 0 or 1) are exactly c * 2^-9, so the
//     byte holding u IS the E4M3 code of u * 2^-9: the conversion spreads
//     nibbles to bytes with two logic ops per four values;
//   * an int8 activation a = 16 hi + lo with hi = (a + 8) >> 4 in [-8, 8]
//     and lo in [-8, 7], both exact in E4M3 (normal codes); a small
//     pre-pass writes A' (2 mp rows: hi rows, then lo rows) and the row sums
//     R[m] = sum_k A[m, k];
//   * sum_k a v = 2^9 (16 S_hi + S_lo) - 8 R[m], where S_hi, S_lo are the
//     fp32 column sums; each is an integer multiple of 2^-9 of magnitude at
//     most 120 K 2^-9 (K <= 32768 keeps the integer part below 2^22), hence
//     exact.
// The converted weights never touch shared memory: converter warps write
// them to tensor memory (tcgen05.st) and the MMA reads its A operand from
// there (swap-AB as in skinny.cu: the 128-row MMA dimension runs over
// weight rows, N = 2 mp over the A' rows).  Inside each group of 8 k the
// converters emit the even k first, then the odd k; the pre-pass writes A'
// in the same order, so the products pair up.
// Work split as in skinny.cu: stream-K over (tile, K block) units.  The
// results are exact integers, so the CTAs sharing a tile simply add their
// int32 shares into D (red.add; integer addition is exact in any order, so
// the result is deterministic): the pre-pass zeroes the columns of D of the
// tiles that are shared, and the CTA holding a tile's first K block also
// adds the row-sum correction.  No partial buffers, counters or fix-up.
//
// Warps: 0 weight producer; 1 MMA issuer and TMEM owner; 2..5 epilogue (one
// per TMEM lane quarter); 6..13 converters (two groups of four, one warp per
// lane quarter in each, taking alternate units); 14 A' producer; 15 second
// MMA issuer.
// Shared memory: a ring of packed-weight slots (128-byte swizzled rows),
// released once the converters have read them, and a ring of A' slots (two
// boxes each), one per converted weight buffer.  TMEM: the accumulators
// (columns 0-255) and four converted weight buffers (256-511); unit i of a
// CTA uses buffer and A' slot i mod 4.  The converters mark a buffer ready
// once its weights are stored and its A' has landed; the MMA that read it
// frees buffer and slot with one commit.
// Two MMA issuers: at these shapes an MMA takes ~25 ns and a single issuing
// thread's per-unit wait, fence and commit leave the tensor pipe idle for
// about as long again; with units alternating between two threads, each
// with its own accumulators, one thread's bookkeeping overlaps the other's
// MMAs.  Each issuer has two accumulators (alternating over segments, so
// the epilogue of one overlaps the next) when 2 mp <= 64, else one.  The epilogue adds the two
// accumulators: each partial sum is an integer multiple of 2^-9 below 2^13
// in magnitude, exact in fp32, and is converted to an integer before the
// addition.
#include <cuda_fp8.h>

#include <cstring>

#include "internal.h"

namespace tmg {
namespace {

constexpr int kTileN = 128;                       // weight rows per tile (MMA M, TMEM lanes)
constexpr int kBK = 256;                          // k per K block
constexpr int kPackedBytes = kTileN * kBK / 2;    // 16 KB: 128 rows x 128 bytes of nibbles
constexpr int kABoxK = 128;                       // k (bytes) per A' box row: one 128-byte swizzle span
constexpr int kWCols = kBK / 4;                   // TMEM columns of E4M3 weights per K block (64)
constexpr int kWBufs = 4;
constexpr int kAccRegion = 256;                   // accumulators: 2 x 128 columns (one issuer) or 4 x 64 (two)
constexpr int kWCol0 = kAccRegion;                // first weight column
constexpr int kTmemCols = 512;
constexpr int kMaxMP = 64;
constexpr int kConvWarps = 8;
constexpr int kFirstConvWarp = 6;
constexpr int kAProducerWarp = kFirstConvWarp + kConvWarps;       // 14
constexpr int kSecondMmaWarp = kAProducerWarp + 1;                // 15
constexpr int kThreads = 32 * (kSecondMmaWarp + 1);               // 512
constexpr int kMaxWStages = 16;
constexpr int kSmemBudget = 225 * 1024;

static_assert(kWCol0 + kWBufs * kWCols <= kTmemCols, "TMEM columns");
static_assert(kTileN == kW4TileN && kBK == kW4BK, "pre-shuffled block shape");

// Two rings in shared memory: weight slots (16 KB of packed weights each),
// freed as soon as the converters have read them, and kWBufs A' slots (two
// boxes of 2 mp rows x 128 bytes), freed with the converted weight buffer
// of the same unit.
__host__ __device__ constexpr int a_box_bytes(int mp) { return 2 * mp * kABoxK; }
__host__ __device__ constexpr int a_stage_bytes(int mp) { return 2 * a_box_bytes(mp); }
__host__ __device__ constexpr int bar_bytes() { return (2 * kMaxWStages + 3 * kWBufs + 8) * 8 + 16; }
int w_stages_for(int mp)
{
    const int s = (kSmemBudget - bar_bytes() - 1024 - kWBufs * a_stage_bytes(mp)) / kPackedBytes;
    return s > kMaxWStages ? kMaxWStages : s;
}
int smem_for(int mp)
{
    return w_stages_for(mp) * kPackedBytes + kWBufs * a_stage_bytes(mp) + bar_bytes() + 1024;
}
constexpr int kIssuers = 2;
// Accumulators per MMA issuer: two when all four (2 mp columns each) fit in
// the accumulator region, else one.
int accs_for(int mp) { return 2 * kIssuers * 2 * mp <= kAccRegion ? 2 : 1; }

__device__ __forceinline__ int seg_end(int kb0, int KB, int64_t left)
{
    return left < static_cast<int64_t>(KB - kb0) ? kb0 + static_cast<int>(left) : KB;
}

// Units go to the two MMA issuers by the parity of the CTA-local unit
// index.  Does issuer j take one of the local units [i0, i1) (non-empty)?
__device__ __forceinline__ bool issuer_has(int64_t i0, int64_t i1, int j)
{
    return i1 - i0 >= 2 || static_cast<int>(i0 & 1) == j;
}

// Accumulator of issuer j for the s-th segment it takes part in, and the
// parity of that accumulator's s-th use (nacc accumulators per issuer).
__device__ __forceinline__ int acc_index(int j, int s, int nacc) { return j * nacc + (nacc == 2 ? (s & 1) : 0); }
__device__ __forceinline__ uint32_t acc_phase(int s, int nacc) { return static_cast<uint32_t>((nacc == 2 ? s >> 1 : s) & 1); }

// Programmatic dependent launch: the pre-pass lets the GEMM start early;
// the GEMM waits for the pre-pass's results only where it reads them.
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Contiguous bulk copy global -> shared with an L2 eviction-priority hint;
// both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load_hint(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T, E4M3 operands, one CTA (kind::f8f6f4,
// K = 32 per instruction: 8 TMEM columns of A per row).
// Issued warp-wide: the elect.sync predicate picks one lane of the issuing
// warp, which runs its loop in warp-uniform control flow.
__device__ __forceinline__ void mma_e4m3_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// registers -> TMEM: 32 lanes x 32 consecutive columns (thread i writes lane
// base + i); complete once tmem_wait_st returns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Position of k (mod 8) inside its group of 8 in the MMA's k order: the even
// k first, then the odd k (the order the converters emit).
__host__ __device__ constexpr int k_slot(int j) { return (j >> 1) + 4 * (j & 1); }

__device__ __forceinline__ int64_t unit_start(int c, int64_t U, int G) { return (static_cast<int64_t>(c) * U) / G; }

// A' (2 mp rows x K, E4M3) and R: blocks m < mp, one per activation row.
// Row m holds the codes of hi = (a + 8) >> 4, row mp + m those of
// lo = a - 16 hi, for a = A[m, k], each group of 8 k in k_slot order; rows
// m >= M are zero.  R[m] = sum_k A[m, k].
// Blocks mp .. mp + kZeroBlocks - 1 zero D (rows < M) in the tiles that the
// GEMM's G CTAs share, which take red.adds: a tile is shared exactly when a
// CTA's first unit c U / G (1 <= c < G) falls inside it, not at its start.
constexpr int kSplitThreads = 256;
constexpr int kZeroBlocks = 16;

__global__ void __launch_bounds__(kSplitThreads)
    split_activations_kernel(const int8_t *__restrict__ A, int M, int N, int K, int mp, uint8_t *__restrict__ Ap,
                             int32_t *__restrict__ R, int32_t *__restrict__ D, int64_t ldd, int G)
{
    griddep_launch_dependents();
    if (blockIdx.x >= mp) {
        const int KB = (K + kBK - 1) / kBK;
        const int64_t U = static_cast<int64_t>((N + kTileN - 1) / kTileN) * KB;
        const int warps = kZeroBlocks * kSplitThreads / 32;
        const int wid = (blockIdx.x - mp) * (kSplitThreads / 32) + threadIdx.x / 32;
        for (int cb = 1 + wid; cb < G; cb += warps) {
            const int64_t b = unit_start(cb, U, G);
            if (b % KB == 0)
                continue;                                      // the boundary is a tile start
            const int64_t t = b / KB;
            for (int col = threadIdx.x % 32; col < kTileN; col += 32) {
                const int64_t n = t * kTileN + col;
                if (n < N)
                    for (int m = 0; m < M; ++m)
                        D[static_cast<int64_t>(m) * ldd + n] = 0;
            }
        }
        return;
    }
    __shared__ int warp_sums[kSplitThreads / 32];
    const int m = blockIdx.x;
    const int groups = K / 8;
    uint8_t *hi_row = Ap + static_cast<int64_t>(m) * K;
    uint8_t *lo_row = Ap + static_cast<int64_t>(mp + m) * K;
    const bool vec = (reinterpret_cast<uintptr_t>(A) & 7u) == 0;    // K is a multiple of 32
    int sum = 0;
#pragma unroll 4
    for (int g = threadIdx.x; g < groups; g += kSplitThreads) {
        int8_t av[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (m < M) {
            const int8_t *src = A + static_cast<int64_t>(m) * K + 8 * g;
            if (vec)
                std::memcpy(av, __builtin_assume_aligned(src, 8), 8);
            else
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    av[j] = src[j];
        }
        uint8_t hc[8], lc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int a = av[j];
            const int hi = (a + 8) >> 4;
            const int lo = a - 16 * hi;
            sum += a;
            hc[k_slot(j)] = __nv_cvt_float_to_fp8(static_cast<float>(hi), __NV_SATFINITE, __NV_E4M3);
            lc[k_slot(j)] = __nv_cvt_float_to_fp8(static_cast<float>(lo), __NV_SATFINITE, __NV_E4M3);
        }
        uint2 hw, lw;
        std::memcpy(&hw, hc, 8);
        std::memcpy(&lw, lc, 8);
        *reinterpret_cast<uint2 *>(hi_row + 8 * g) = hw;
        *reinterpret_cast<uint2 *>(lo_row + 8 * g) = lw;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    if (threadIdx.x % 32 == 0)
        warp_sums[threadIdx.x / 32] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int total = 0;
        for (int w = 0; w < kSplitThreads / 32; ++w)
            total += warp_sums[w];
        R[m] = total;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    w4a8_skinny_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA,
                       const uint8_t *__restrict__ Bs, int32_t *__restrict__ D, int64_t ldd,
                       const int32_t *__restrict__ R, int M, int N, int K, int mp, int wstages, int nacc,
                       ErrCtx err)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);   // weight ring
    const int abytes = a_stage_bytes(mp);
    uint8_t *aring = smem + wstages * kPackedBytes;                     // A' ring
    uint64_t *wfull = reinterpret_cast<uint64_t *>(aring + kWBufs * abytes);
    uint64_t *wempty = wfull + kMaxWStages;
    uint64_t *afull = wempty + kMaxWStages;
    uint64_t *cready = afull + kWBufs;                         // weights in TMEM and A' landed (converters)
    uint64_t *cfree = cready + kWBufs;                         // buffer and A' slot consumed (MMA commit)
    uint64_t *tfull = cfree + kWBufs;                          // per accumulator
    uint64_t *tempty = tfull + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int G = gridDim.x, c = blockIdx.x;
    const int tiles = (N + kTileN - 1) / kTileN;
    const int KB = (K + kBK - 1) / kBK;                        // a ragged last K block reads zeros
    const int64_t U = static_cast<int64_t>(tiles) * KB;
    const int64_t u_begin = unit_start(c, U, G), u_end = unit_start(c + 1, U, G);
    const int abox = a_box_bytes(mp);

    if (threadIdx.x == 0) {
        for (int s = 0; s < wstages; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], kConvWarps / 2);             // the converter group of the unit
        }
        for (int b = 0; b < kWBufs; ++b) {
            mbar_init(&afull[b], 1);
            mbar_init(&cready[b], kConvWarps / 2);
            mbar_init(&cfree[b], 1);                           // the MMA commit
        }
        for (int b = 0; b < 4; ++b) {
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

    const int64_t n_units = u_end - u_begin;
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------ weight producer
            // The weights do not depend on the pre-pass.  Unit u's weights:
            // the pre-shuffled block u (16 KB, contiguous), else a 128 x
            // 128-byte box of the row-major B.
            const uint64_t stream_b = policy_evict_first();  // the weights are read once
            int64_t issued = 0;
            for (int64_t i = 0; i < n_units; ++i) {
                const int ws = static_cast<int>(i % wstages);
                const uint32_t ph = static_cast<uint32_t>((i / wstages) & 1);
                if (!mbar_wait(&wempty[ws], ph ^ 1u, err, abort_flag, kSiteProducerEmpty))
                    break;
                const int64_t u = u_begin + i;
                uint8_t *st = smem + ws * kPackedBytes;
                mbar_arrive_expect_tx(&wfull[ws], kPackedBytes);
                if (Bs)
                    bulk_load_hint(st, Bs + u * kPackedBytes, kPackedBytes, &wfull[ws], stream_b);
                else
                    tma_load_2d_hint(st, &tmB, &wfull[ws], static_cast<int>(u % KB) * (kBK / 2),
                                     static_cast<int>(u / KB) * kTileN, stream_b);
                ++issued;
            }
            // before leaving, let every load this thread requested land
            for (int64_t i = issued - 1; i >= 0 && i >= issued - wstages; --i)
                mbar_wait(&wfull[i % wstages], static_cast<uint32_t>((i / wstages) & 1), err, nullptr, kSiteDrain);
        }
    } else if (warp == kAProducerWarp) {
        if (lane == 0) {
            // ---------------------------------------------- A' producer
            const uint64_t keep_a = policy_evict_last();    // A' is re-read by every CTA
            griddep_wait();                                  // A' comes from the pre-pass
            int64_t issued = 0;
            for (int64_t i = 0; i < n_units; ++i) {
                // slot i mod kWBufs is free once the MMAs of unit i - kWBufs
                // (which used the same converted weight buffer) completed
                const int as = static_cast<int>(i % kWBufs);
                const uint32_t ph = static_cast<uint32_t>((i / kWBufs) & 1);
                if (!mbar_wait(&cfree[as], ph ^ 1u, err, abort_flag, kSiteProducerEmpty))
                    break;
                const int kb = static_cast<int>((u_begin + i) % KB);
                uint8_t *st = aring + as * abytes;
                mbar_arrive_expect_tx(&afull[as], static_cast<uint32_t>(abytes));
                tma_load_2d_hint(st, &tmA, &afull[as], kb * kBK, 0, keep_a);
                tma_load_2d_hint(st + abox, &tmA, &afull[as], kb * kBK + kABoxK, 0, keep_a);
                ++issued;
            }
            for (int64_t i = issued - 1; i >= 0 && i >= issued - kWBufs; --i)
                mbar_wait(&afull[i % kWBufs], static_cast<uint32_t>((i / kWBufs) & 1), err, nullptr, kSiteDrain);
        }
    } else if (warp == 1 || warp == kSecondMmaWarp) {
        const int j = warp == 1 ? 0 : 1;                       // issuer index
        // ---------------------------------------------------- MMA issuers
        // MMA A = converted weights (TMEM, 128 rows), MMA B = A' (2 mp
        // rows).  Issuer j takes the units i with i mod 2 = j into its
        // own accumulators (acc_index: one, or two alternating over the
        // segments it has units in).  The whole warp runs the loop; one
        // elected lane issues.
        const uint32_t idesc = idesc_e4m3_f32(kTileN, 2 * mp);
        const int acc_cols = kAccRegion / (kIssuers * nacc);
        int64_t i0 = 0;                                    // local index of the segment's first unit
        int nseg = 0;                                      // segments this issuer took part in
        bool ok = true;
        for (int64_t u = u_begin; u < u_end && ok;) {
            const int kb0 = static_cast<int>(u % KB);
            const int kb1 = seg_end(kb0, KB, u_end - u);
            const int64_t i1 = i0 + (kb1 - kb0);
            if (issuer_has(i0, i1, j)) {
                const int acc = acc_index(j, nseg, nacc);
                if (!mbar_wait_warp(&tempty[acc], acc_phase(nseg, nacc) ^ 1u, err, abort_flag, kSiteMmaTmemEmpty))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * acc_cols;
                bool first = true;
                for (int64_t i = i0 + (static_cast<int>(i0 & 1) != j ? 1 : 0); i < i1; i += kIssuers) {
                    const int wb = static_cast<int>(i % kWBufs);
                    if (!mbar_wait_warp(&cready[wb], static_cast<uint32_t>((i / kWBufs) & 1), err, abort_flag,
                                        kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_src = tmem_base + kWCol0 + wb * kWCols;
                    const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(aring + wb * abytes));
                    const uint64_t bdesc1 = sdesc_kmajor_sw128(smem_u32(aring + wb * abytes + abox));
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k) {
                        const uint64_t bdesc =
                            (k < 4 ? bdesc0 : bdesc1) + static_cast<uint64_t>(((k & 3) * 32) >> 4);
                        mma_e4m3_ts_w(d_tmem, a_src + 8 * k, bdesc, idesc, !first || (k != 0));
                    }
                    first = false;
                    mma_commit_w(&cfree[wb]);
                }
                if (!ok)
                    break;
                mma_commit_w(&tfull[acc]);
                ++nseg;
            }
            i0 = i1;
            u += kb1 - kb0;
        }
    } else if (warp >= kFirstConvWarp) {
        // ------------------------------------------------- converters
        // Thread = weight row r of the tile = TMEM lane r.  The two groups
        // of four warps (one per TMEM lane quarter in each) take alternate
        // units: per unit a warp reads its row's 8 swizzled 16-byte chunks,
        // releases the staging slot, spreads the nibbles to offset-binary
        // E4M3 bytes and stores the unit's 64 TMEM columns of its lane
        // quarter with one wait, so each warp's per-unit waits and store
        // latency are paid once per two units.
        const int q = warp & 3;
        const int grp = (warp - kFirstConvWarp) >> 2;
        const int r = q * 32 + lane;
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kWCol0;
        int ws = grp, wb = grp;                                // unit i: slot i mod wstages, buffer i mod kWBufs
        uint32_t phase = 0, wphase = 0;
        for (int64_t i = grp; i < n_units; i += 2) {
            if (!mbar_wait(&wfull[ws], phase, err, abort_flag, kSiteMmaFull) ||
                !mbar_wait(&cfree[wb], wphase ^ 1u, err, abort_flag, kSiteProducerEmpty))
                break;
            tc_fence_after();
            const uint8_t *src = smem + ws * kPackedBytes + r * 128;
            uint4 w[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                w[c] = *reinterpret_cast<const uint4 *>(src + ((c ^ (r & 7)) << 4));
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&wempty[ws]);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t out[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = w[4 * hh + c];
                    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t y = words[j] ^ 0x88888888u;   // offset binary: v + 8
                        out[8 * c + 2 * j] = y & 0x0F0F0F0Fu;       // even k
                        out[8 * c + 2 * j + 1] = (y >> 4) & 0x0F0F0F0Fu;   // odd k
                    }
                }
                tmem_st32(t_row + wb * kWCols + 32 * hh, out);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            // the MMA issuer waits on this barrier alone: the unit's A'
            // arrival is folded into it
            int landed = 1;
            if (lane == 0) {
                landed = mbar_wait(&afull[wb], wphase, err, abort_flag, kSiteMmaFull) ? 1 : 0;
                if (landed)
                    mbar_arrive(&cready[wb]);
            }
            if (!__shfl_sync(0xFFFFFFFFu, landed, 0))
                break;
            if ((ws += 2) >= wstages) {
                ws -= wstages;
                phase ^= 1u;
            }
            if ((wb += 2) >= kWBufs) {
                wb -= kWBufs;
                wphase ^= 1u;
            }
        }
    } else {
        // -------------------------------------------------- epilogue
        // thread owns weight row n_local = 32 q + lane; in each accumulator
        // TMEM columns m and mp + m hold the hi and lo sums of activation row
        // m (scaled 2^-9); the issuers' shares of a segment are added
        const int q = warp & 3;
        const int n_local = q * 32 + lane;
        const int acc_cols = kAccRegion / (kIssuers * nacc);
        griddep_wait();                                        // R comes from the pre-pass
        int64_t i0 = 0;
        int nseg0 = 0, nseg1 = 0;                              // segments each issuer took part in
        bool ok = true;
        for (int64_t u = u_begin; u < u_end && ok;) {
            const int tile = static_cast<int>(u / KB);
            const int kb0 = static_cast<int>(u % KB);
            const int kb1 = seg_end(kb0, KB, u_end - u);
            const int64_t i1 = i0 + (kb1 - kb0);
            u += kb1 - kb0;
            int32_t v[kMaxMP];
#pragma unroll
            for (int m = 0; m < kMaxMP; ++m)
                v[m] = 0;
            for (int j = 0; j < kIssuers; ++j) {
                if (!issuer_has(i0, i1, j))
                    continue;
                const int ns = j == 0 ? nseg0++ : nseg1++;
                const int acc = acc_index(j, ns, nacc);
                if (!mbar_wait(&tfull[acc], acc_phase(ns, nacc), err, abort_flag, kSiteEpiTmemFull)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                tc_fence_after();
                const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * acc_cols;
#pragma unroll
                for (int ch = 0; ch < kMaxMP / 16; ++ch) {
                    if (ch * 16 < mp) {
                        uint32_t h[16], l[16];
                        tmem_ld16(tb + ch * 16, h);
                        tmem_ld16(tb + mp + ch * 16, l);
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            v[ch * 16 + t] += 16 * __float2int_rn(__uint_as_float(h[t]) * 512.0f) +
                                              __float2int_rn(__uint_as_float(l[t]) * 512.0f);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&tempty[acc]);
            }
            i0 = i1;
            if (!ok)
                break;

            const int n = tile * kTileN + n_local;
            int32_t *d = D + n;
            const int64_t d_limit = static_cast<int64_t>(M - 1) * ldd + N;     // elements of D
            if (n < N && kb0 == 0 && kb1 == KB) {
                // the whole tile is this CTA's: plain stores
#pragma unroll
                for (int m = 0; m < kMaxMP; ++m)
                    if (m < M && bounds_ok(static_cast<int64_t>(m) * ldd + n, d_limit, err, kBndStoreD))
                        d[static_cast<int64_t>(m) * ldd] = v[m] - 8 * R[m];
            } else if (n < N) {
                // a share of a tile: add into the zeroed D; the first K
                // block's holder adds the correction too
                const int corr = kb0 == 0 ? 8 : 0;
#pragma unroll
                for (int m = 0; m < kMaxMP; ++m)
                    if (m < M && bounds_ok(static_cast<int64_t>(m) * ldd + n, d_limit, err, kBndStoreD))
                        atomicAdd(d + static_cast<int64_t>(m) * ldd, v[m] - corr * R[m]);
            }
            __syncwarp();
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

// Pre-shuffled weights ("FlyDSL Kernel Authoring Skill", §6 GEMM Pattern
// (Preshuffle): B rearranged once so that the kernel's tiles are
// contiguous).  Block (t, kb) = 128 weight rows x 256 k, 16 KB, sits at
// ((t * KB) + kb) * 16 KB: row r's 128 bytes at r * 128, its 16-byte chunk
// c (k = kb * 256 + 32 c .. + 31, even k in the low nibble) at chunk slot
// c XOR (r mod 8) — exactly the image the 128-byte swizzled tensor-map load
// leaves in shared memory.  Rows past N and chunks past K are zero.  One
// thread per 16-byte chunk; K a multiple of 32, so a chunk is either whole
// or entirely past K.
__global__ void __launch_bounds__(256)
    w4a8_preshuffle_kernel(const uint8_t *__restrict__ B, int64_t N, int64_t K, uint8_t *__restrict__ Bs,
                           int64_t chunks)
{
    const int64_t KB = (K + kBK - 1) / kBK;
    const int64_t row_bytes = K / 2;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t blk = i / (kTileN * 8);
        const int r = static_cast<int>((i / 8) % kTileN);
        const int slot = static_cast<int>(i % 8);
        const int64_t n = (blk / KB) * kTileN + r;
        const int64_t byte0 = (blk % KB) * (kBK / 2) + 16 * (slot ^ (r & 7));
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < N && byte0 < row_bytes)
            v = *reinterpret_cast<const uint4 *>(B + n * row_bytes + byte0);
        *reinterpret_cast<uint4 *>(Bs + 16 * i) = v;
    }
}

}  // namespace

size_t w4a8_preshuffled_bytes(int64_t N, int64_t K)
{
    return static_cast<size_t>((N + kTileN - 1) / kTileN) * static_cast<size_t>((K + kBK - 1) / kBK) * kPackedBytes;
}

cudaError_t launch_w4a8_preshuffle(const void *B, int64_t N, int64_t K, void *Bs, int num_sms, cudaStream_t s)
{
    const int64_t chunks = static_cast<int64_t>(w4a8_preshuffled_bytes(N, K) / 16);
    int64_t blocks = (chunks + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    note_launch();
    w4a8_preshuffle_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint8_t *>(B), N, K,
                                                                        static_cast<uint8_t *>(Bs), chunks);
    return cudaGetLastError();
}

int w4a8_skinny_grid(int64_t N, int64_t K, int num_sms)
{
    const int64_t units = ((N + kTileN - 1) / kTileN) * ((K + kBK - 1) / kBK);
    return static_cast<int>(units < num_sms ? units : num_sms);
}

cudaError_t launch_w4a8_skinny(const W4a8SkinnyArgs &a, const ErrCtx &err, cudaStream_t s)
{
    // the activation split (one block per A' row pair), then the GEMM as a
    // programmatic dependent launch: its set-up and first weight loads
    // overlap the split
    note_launch();
    split_activations_kernel<<<static_cast<unsigned>(a.mp + kZeroBlocks), kSplitThreads, 0, s>>>(
        static_cast<const int8_t *>(a.A), a.M, a.N, a.K, a.mp, a.Ap, a.R, a.D, a.ldd, a.grid);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int wstages = w_stages_for(a.mp), nacc = accs_for(a.mp);
    const int smem = smem_for(a.mp);
    if ((e = ensure_smem_attr(reinterpret_cast<const void *>(w4a8_skinny_kernel), smem)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_launch();
    return cudaLaunchKernelEx(&cfg, w4a8_skinny_kernel, a.tmB, a.tmA, a.Bs, a.D, a.ldd,
                              static_cast<const int32_t *>(a.R), a.M, a.N, a.K, a.mp, wstages, nacc, err);
}

}  // namespace tmg
