// mx_common.cuh — pieces shared by the one-CTA and CTA-pair MXFP4 kernels:
// the block-scaled instruction descriptor, the scale-chunk copy into TMEM,
// and the layout of the relaid scales.
//
// Scales of one operand are relaid (pre-pass, mx_scale_relayout in mxfp4.cu)
// into groups of `group_rows` rows (the rows one CTA or one pair tile
// consumes); for each group and each 256-element K block there are
// nsub = ceil(group_rows / 128) sub-blocks of 128 rows, each two 512-byte
// chunks; chunk c holds K-blocks 4c..4c+3, and its 16-byte line r0 (0..31)
// holds the scales of sub-block rows r0, r0+32, r0+64, r0+96 — the order in
// which TMEM must hold them (lane = row mod 32 in every lane quarter,
// column = row / 32, byte = K-block) for the block-scaled MMA.
//   compact form (one-CTA kernel): per (group, K block) the nsub sub-blocks
//     of 1 KB, [chunk 0][chunk 1] each; copied with 32x128b.warpx4.
//   wide form (pair kernel): per (group, K block) nsub x 4 KB; wide copy p
//     (p < nsub) takes the 4 KB at p x 4 KB = [X x4][Y x4], the chunks for
//     its columns 0-3 and 4-7: (chunk 0, chunk 1) of the one sub-block when
//     nsub = 1, (sub-block 0, sub-block 1) of chunk p when nsub = 2.
#pragma once

#include "internal.h"

namespace tmg {
namespace mx {

constexpr int kBK = 256;          // K elements per K block (128 bytes of codes)
constexpr int kBKBytes = 128;
constexpr int kSfChunk = 512;     // 32 lines x 16 bytes
constexpr int kSfBlock = 1024;    // one 128-row sub-block: 2 chunks

// Shared-memory descriptor without swizzle (8-row x 16-byte core matrices,
// stride byte offset 128 between consecutive 8-row groups), for tcgen05.cp.
__device__ __forceinline__ uint64_t sdesc_noswizzle_rows16(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 16;
    d |= static_cast<uint64_t>(128 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Instruction descriptor, kind::mxf4 block-scaled: B scale id (bits 4-5),
// A format (7-9) = 1 (E2M1), B format (10-12) = 1 (E2M1), K-major A and B,
// N >> 3 (17-22), scale type (23) = 1 (E8M0), M >> 4 (24-28), A scale id
// (29-30), K size (31) = 0 (64 dense).  The id selects the two scales inside
// each 32-bit TMEM column: 0 -> bytes 0-1, 2 -> bytes 2-3.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, uint32_t sf_id)
{
    return (sf_id << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | (sf_id << 29);
}

// Wide copies: 128 lanes x 32 bytes (8 TMEM columns) per instruction.  Each
// tcgen05.cp costs the tensor pipe about the same whatever its width, so the
// pair kernel moves its scales with these: the source holds, for lane l, the
// 16-byte line (l mod 32) of two chunks — i.e. each 512-byte chunk repeated
// four times — as two 2 KB halves (columns 0-3 from the first, 4-7 from the
// second).  Descriptor: no swizzle, 8-row x 16-byte core matrices 128 bytes
// apart, the two 16-byte column halves 2 KB apart.
constexpr int kWideSrcBytes = 4096;

__device__ __forceinline__ uint64_t sdesc_wide_scales(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(2048 >> 4) << 16;     // leading byte offset: next 16-byte column half
    d |= static_cast<uint64_t>(128 >> 4) << 32;      // stride byte offset: next 8-row group
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Warp-wide forms (elect.sync predicate on the instruction; see the
// warp-wide MMA issue notes beside mma_bf16_w): the issuing loops run on a
// whole warp and one elected lane issues.
__device__ __forceinline__ void mma_mxf4_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X "
        "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_mxf4_pair_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X "
        "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy one 512-byte scale chunk (32 lines x 16 bytes) from shared memory to
// 4 TMEM columns, replicated into all four lane quarters.
__device__ __forceinline__ void tmem_cp_chunk_w(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// The same, issued by CTA 0 of a pair for both CTAs (each CTA's chunk at the
// same shared-memory offset goes to that CTA's TMEM).
__device__ __forceinline__ void tmem_cp_chunk_pair_w(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// One wide copy (128 lanes x 32 bytes, the layout of sdesc_wide_scales) for
// both CTAs of a pair.
__device__ __forceinline__ void tmem_cp_wide_pair_w(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.cp.cta_group::2.128x256b [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// Programmatic dependent launch: the relayout pre-pass lets the GEMM start
// early; the GEMM waits for the pre-pass's results only where it reads them.
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace mx
}  // namespace tmg
