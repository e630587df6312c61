// device.cuh — sm_103a building blocks written as inline PTX: mbarriers,
// TMA tile loads, TMEM allocation, tcgen05 MMA / commit / load, shared-memory
// matrix descriptors, and a bounded barrier wait that reports instead of
// hanging.
//
// These play the part that copy atoms and MMA atoms play on the FlyDSL pages
// ("add-target-atom-op", §1.1 two-level type design: a generic atom wrapping
// one concrete instruction): here each helper issues exactly one PTX
// instruction of the Blackwell tensor-core / TMA families.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tmg {

// Device error word codes (OR-ed into the word, high byte = kind).
enum : uint32_t {
    kErrTimeout = 0x01000000u,
    kErrBounds = 0x02000000u,     // debug build: an offset outside its buffer (site in the low bits)
};

// Wait-site identifiers (low bits of the error word) for diagnostics.
enum : uint32_t {
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaTmemEmpty = 3,
    kSiteEpiTmemFull = 4,
    kSiteDrain = 5,
    kSiteProbe = 6,
    // bounds-check sites of the debug build
    kBndStoreD = 16,        // a store of D
    kBndPartials = 17,      // split-K / stream-K partial sums
    kBndCounters = 18,      // split-K / stream-K tile counters
    kBndScratch = 19,       // other library scratch (W4A8 split activations and row sums)
    kBndProbe = 20,         // tmg_debug_bounds_probe
};

// Arguments every kernel receives for error reporting.
struct ErrCtx {
    uint32_t *word;          // device error word (static device memory)
    uint64_t budget_ns;      // budget of one bounded wait
};

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarriers

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait until the phase with the given parity of `bar` has completed.  Gives
// up after ctx.budget_ns (or if *abort becomes non-zero): records the site in
// the device error word, raises *abort so the CTA's other roles stop too,
// and returns false.  Never spins without limit.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const ErrCtx &ctx,
                                          volatile int *abort, uint32_t site)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (abort && *abort)
                return false;
            if (globaltimer() - t0 > ctx.budget_ns || it > 0x7FFFFFF0u) {
                atomicOr(ctx.word, kErrTimeout | site);
                if (abort)
                    *abort = 1;
                return false;
            }
        }
    }
}

// --------------------------------------------------- debug bounds checks
//
// Built with -DTMG_DEBUG_BOUNDS (build.py, debug build: libtmg_debug.so),
// every store of D and every access to split-K / stream-K scratch in the GEMM
// kernels first checks its computed element offset against the extent of
// its buffer: an offset outside [0, limit) ORs kErrBounds | site into the
// device error word and the access is skipped, so tmg_check reports it
// instead of memory being overwritten.  In the normal build the check is a
// constant `true` and costs nothing.  (TMA loads and stores need no check:
// the hardware clips them to the tensor map's extents.)
__device__ __forceinline__ bool bounds_ok(int64_t off, int64_t limit, const ErrCtx &err, uint32_t site)
{
#ifdef TMG_DEBUG_BOUNDS
    if (off < 0 || off >= limit) {
        atomicOr(err.word, kErrBounds | site);
        return false;
    }
#else
    (void)off;
    (void)limit;
    (void)err;
    (void)site;
#endif
    return true;
}

// The same for the n elements off .. off + n - 1 of one vector access (an
// empty span, n <= 0, touches nothing).
__device__ __forceinline__ bool span_ok(int64_t off, int n, int64_t limit, const ErrCtx &err, uint32_t site)
{
    return n <= 0 || (bounds_ok(off, limit, err, site) && bounds_ok(off + n - 1, limit, err, site));
}

// ------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Same, with an L2 eviction-priority hint (createpolicy result).
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map,
                                                 uint64_t *bar, int32_t c0, int32_t c1,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------ TMEM

// Whole warp: allocate `ncols` TMEM columns (power of two, 32..512); the
// TMEM address is written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// --------------------------------------------------------- tcgen05 MMA

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row / 1024-byte swizzle atoms
// stacked along the row dimension).  Fields: start address >> 4 (bits
// 0-13), leading byte offset >> 4 (16-29; unused for this layout, set to
// 1), stride byte offset >> 4 (32-45; 1024 bytes between 8-row groups),
// fixed 0b001 (46-48), base offset 0 (49-51), relative LBO mode (52),
// swizzle mode 2 = 128B (61-63).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and f32 D, both operands
// K-major, dense: D format (bits 4-5) = 1 (f32), A format (7-9) = 1 (bf16),
// B format (10-12) = 1 (bf16), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with E4M3 A/B and f32 D, both
// operands K-major, dense: D format (bits 4-5) = 1 (f32), A and B formats
// (7-9, 10-12) = 0 (E4M3), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
// One instruction covers K = 32 (32 bytes of each operand row).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N)
{
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// TMEM -> registers: 32 lanes x 32 consecutive 32-bit columns; thread i of
// the warp receives lane (lane base + i).  Waits for completion before
// returning so the registers are safe to use.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 16 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// ------------------------------------------------- CTA pairs (clusters)
//
// Two CTAs of a cluster can run one MMA together (cta_group::2): the MMA
// covers 256 rows, rows 0-127 from CTA 0's shared memory and 128-255 from
// CTA 1's at the same offset; B's N rows are split the same way; each CTA's
// TMEM holds its own 128 rows of the accumulator.  CTA 0 issues the MMAs.

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Whole-cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (any CTA).
// Used by epilogue warps to hand an accumulator back to the MMA issuer: what
// they must have finished is their tcgen05.ld, which tcgen05.wait::ld has
// already completed, so the release is CTA-scoped.  A cluster-scoped release
// would also wait for the warp's earlier global stores to be ordered at
// cluster scope, about a microsecond per arrive on the issuer's critical path.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// mbar_wait for a barrier that other CTAs of the cluster arrive on
// (cluster-scope acquire); same bounded contract as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, const ErrCtx &ctx,
                                                  volatile int *abort, uint32_t site)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (abort && *abort)
                return false;
            if (globaltimer() - t0 > ctx.budget_ns || it > 0x7FFFFFF0u) {
                atomicOr(ctx.word, kErrTimeout | site);
                if (abort)
                    *abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait_cluster_warp(uint64_t *bar, uint32_t parity, const ErrCtx &ctx,
                                                       volatile int *abort, uint32_t site)
{
    return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, ctx, abort, site));
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ------------------------------------------------- warp-wide MMA issue
//
// The MMA-issuing loops run on a whole warp in warp-uniform control flow;
// the tcgen05 instruction itself carries an elect.sync predicate, so exactly
// one lane (the lowest, the same one every time in a converged warp) issues
// it and no branch splits the warp.  Issued from inside a one-lane branch
// instead, a tcgen05.mma was measured at ~70 ns apiece on this part whatever
// its shape, against ~37 ns (N <= 128) and the pipe's own ~66 ns at N = 256
// from the warp-wide loop: inside the branch every operand has to leave the
// uniform datapath before each instruction.  The commits go through the same
// elected lane, so they track exactly the MMAs it issued.

// Every lane waits; the warp leaves together with one agreed result.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, const ErrCtx &ctx,
                                               volatile int *abort, uint32_t site)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx, abort, site));
}

// D[tmem] (+)= A[smem] · B[smem]ᵀ, one tcgen05.mma of the CTA (cta_group::1).
__device__ __forceinline__ void mma_bf16_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation the elected lane issued
// so far has completed.
__device__ __forceinline__ void mma_commit_w(uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// One pair MMA (M = 256) issued by CTA 0.
__device__ __forceinline__ void mma_bf16_pair_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same for E4M3 operands (kind::f8f6f4, K = 32 per instruction).
__device__ __forceinline__ void mma_e4m3_pair_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at this shared-memory offset in every CTA of
// `cta_mask` when the pair's prior tcgen05 operations have completed.
__device__ __forceinline__ void mma_commit_pair_w(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Producer-side counterparts: the loop runs on the whole warp, one elected
// lane announces the bytes and issues the copies.
__device__ __forceinline__ void mbar_arrive_expect_tx_w(uint64_t *bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// 2-D tiled bulk tensor copy global -> shared, completion counted in bytes on
// `bar`; c0 is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d_w(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                              int32_t c1)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// The same into this CTA's shared memory, completion counted on an mbarrier
// that may live in the peer CTA of a pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair_w(void *smem_dst, const CUtensorMap *map, uint32_t bar_cluster_addr,
                                                   int32_t c0, int32_t c1)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint_w(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                                   int32_t c1, uint64_t policy)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// Contiguous bulk copy global -> shared (`bytes` a multiple of 16, both
// addresses 16-byte aligned), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load_w(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 32-byte vector store to global memory (`p` 32-byte aligned): one whole
// 32-byte sector per thread, where two 16-byte stores would write each sector
// in halves.
__device__ __forceinline__ void st_global_v8(void *p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                             uint32_t a5, uint32_t a6, uint32_t a7)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2),
                 "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

// Two fp32 -> packed bf16x2, round to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace tmg
