// internal.h — declarations shared by the library's translation units
// (host launchers of each kernel family and the argument structs they take).
// Not part of the public ABI; see include/tmg.h for that.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"

namespace tmg {

// A rank-2 layout as the kernels see it (same meaning as tmg_layout).
struct DevLayout {
    int32_t depth[2];
    int64_t shape[2][2];
    int64_t stride[2][2];
};

// ---------------------------------------------------------------- FFMA path
struct FfmaArgs {
    const void *A;
    const void *B;
    void *D;
    DevLayout la, lb, ld;
    int64_t M, N, K;
};
// dtype: 0 = f32, 1 = bf16.  Returns the launch status.
cudaError_t launch_ffma(const FfmaArgs &a, int dtype, int num_sms, const ErrCtx &err,
                        cudaStream_t s);

// Skinny CUDA-core path: A (M,K) and B (N,K) bf16 K-major (row strides lda,
// ldb), D (M,N) bf16 row-major with leading dimension ldd; M <= 16.
struct SkinnyFfmaArgs {
    const void *A;
    const void *B;
    void *D;
    int64_t M, N, K, lda, ldb, ldd;
};
cudaError_t launch_skinny_ffma(const SkinnyFfmaArgs &a, int num_sms, cudaStream_t s);

// Fill the (M,N) output with zeros through its layout (K == 0).
cudaError_t launch_zero_fill(void *D, const DevLayout &ld, int64_t M, int64_t N, int dtype,
                             cudaStream_t s);

// ------------------------------------------------------ tcgen05 bf16 path
struct TcArgs {
    CUtensorMap tmA;   // A (M,K) bf16 K-major, box {64, 128}, 128B swizzle
    CUtensorMap tmB;   // B (N,K) bf16 K-major, box {64, BN} (pair kernel: {64, BN/2}), 128B swizzle
    void *D;           // bf16 (M,N), row stride ldd elements, unit column stride
    int64_t ldd;
    int M, N, K;
    int bn;            // tile width (N per tile)
    int kb_elems;      // pair kernel: elements per K block, 64 (bf16) or 128 (E4M3); 0 means 64
    // pair kernel schedule (tc2_plan) and its stream-K scratch
    int pairs;         // clusters launched
    int dp_tiles;      // tiles run data-parallel
    int sk_tiles;      // tiles after them, run stream-K
    int group_m;       // M-tiles per group of the tile order (8 or 16)
    float *partials;   // tc2_partials_bytes()
    uint32_t *counters;  // tc2_counters_bytes(), zero on entry
    int maj;           // pair kernel, bf16: bit 0 A MN-major (tmA over Aᵀ, box {64, 64}), bit 1 B MN-major
                       // (tmB over Bᵀ, box {64, 64}; bn 256 or 128)
};
cudaError_t launch_tc_bf16(const TcArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s);
// One-CTA tile width (64, 128 or 256) for an M x N x K product and its
// estimated time in ns, on the same footing as tc2_pick_bn's estimate.
int tc_pick_bn(int64_t M, int64_t N, int64_t K, int num_sms, double *est_ns);
// CTA-pair variant (cta_group::2, 256 x bn tiles; bn in {256, 224, 192, 128},
// tmB box {64, bn/2}).  Call tc2_plan first, then provide the scratch.
cudaError_t launch_tc2_bf16(const TcArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s);
// Pair-tile width for an M x N x K product (64-element K blocks), from the
// widths 256 / 224 / 192 / 128; tc2_pick_bn_of chooses among `cands` for
// K blocks of kb_elems elements.  The same cost model decides, in
// tc2_plan, between a data-parallel schedule and a stream-K tail.
int tc2_pick_bn(int64_t M, int64_t N, int64_t K, int num_sms, double *est_ns = nullptr);
int tc2_pick_bn_of(int64_t M, int64_t N, int64_t K, int kb_elems, int num_sms, const int *cands, int nc);

// Fused epilogue of the pair kernel: D = bf16(act(acc * scale_a[m] *
// scale_b[n] + bias[n])); scale_a / scale_b may be null (factor 1), bias is
// read only by the bias_* epilogues.
enum { kEpiNone = 0, kEpiBias = 1, kEpiBiasRelu = 2, kEpiBiasSilu = 3, kEpiBiasGelu = 4 };
struct Tc2Epi {
    const float *scale_a;
    const float *scale_b;
    const float *bias;
    int epi;
    int out_i32;       // 0: bf16 D; 1: int32 D = round(y); 2: int32 D += round(y) (no TMA stores)
};
// Pair kernel with the fused epilogue (tc2_fused.cu); bf16 or E4M3 inputs
// (tmA/tmB over bytes for E4M3, box {128, rows}; a.kb_elems = 128);
// a.bn one of kTc2FusedWidths.  Call tc2_plan first, then provide the
// scratch.
cudaError_t launch_tc2_fused(const TcArgs &a, const Tc2Epi &e, bool in_e4m3, const ErrCtx &err,
                             cudaStream_t s);
extern const int kTc2FusedWidths[4];
// W4A8 operands: A (M, K) int8 and B (N, K/2) packed int4 unpacked to bf16
// (M, ldp) and (N, ldp), zero-padded past K; ldp a multiple of 8.
cudaError_t launch_unpack_w4a8(const void *A, const void *B, int64_t M, int64_t N, int64_t K, void *PA, void *PB,
                               int64_t ldp, int num_sms, cudaStream_t s, bool b_preshuffled = false);
// Decode-shaped W4A8 (w4a8_skinny.cu): M <= 64, K a multiple of 32 and at
// most 32768.  tmB: packed weights (N, K/2) u8, box {128, 128}, 128-byte
// swizzle; tmA: the split activations A' (2 mp, K) E4M3 (written by the
// launch's pre-pass into Ap), box {128, 2 mp}, 128-byte swizzle.
struct W4a8SkinnyArgs {
    CUtensorMap tmB;
    CUtensorMap tmA;
    const void *A;        // (M, K) int8
    uint8_t *Ap;          // scratch: 2 mp x K bytes
    int32_t *R;           // scratch: mp row sums of A
    const uint8_t *Bs;    // pre-shuffled weights, or null: read B through tmB
    int32_t *D;           // (M, N) int32 row-major, row stride ldd
    int64_t ldd;
    int M, N, K, mp;
    int grid;
};
int w4a8_skinny_grid(int64_t N, int64_t K, int num_sms);

// Pre-shuffled W4A8 weights: block (t, kb) of 128 rows x 256 k (16 KB) at
// (t * KB + kb) * 16 KB, KB = ceil(K / 256); row r's 128 bytes at r * 128,
// its 16-byte chunk c at chunk slot c XOR (r mod 8); K a multiple of 32.
constexpr int kW4TileN = 128;
constexpr int kW4BK = 256;
size_t w4a8_preshuffled_bytes(int64_t N, int64_t K);
cudaError_t launch_w4a8_preshuffle(const void *B, int64_t N, int64_t K, void *Bs, int num_sms, cudaStream_t s);

// Offset in the pre-shuffled image of the 4 bytes holding k0 .. k0 + 7 of
// weight row n (k0 a multiple of 8).
__host__ __device__ inline int64_t w4a8_preshuffled_offset(int64_t n, int64_t k0, int64_t KB)
{
    const int64_t r = n % kW4TileN;
    const int64_t byte = (k0 % kW4BK) / 2;
    return (((n / kW4TileN) * KB + k0 / kW4BK) * kW4TileN + r) * 128 + 16 * ((byte / 16) ^ (r & 7)) + byte % 16;
}
cudaError_t launch_w4a8_skinny(const W4a8SkinnyArgs &a, const ErrCtx &err, cudaStream_t s);

// D[m,n] = bf16(act(bias[n])) (or 0 without a bias): the fused GEMM at K = 0.
cudaError_t launch_fused_k0(void *D, int64_t M, int64_t N, const Tc2Epi &e, cudaStream_t s);
// Fill pairs / dp_tiles / sk_tiles for a.M, a.N, a.K, a.bn: data-parallel,
// or a stream-K tail where the cost model expects it to pay.
void tc2_plan(TcArgs &a, int num_sms);
size_t tc2_partials_bytes(const TcArgs &a);
size_t tc2_counters_bytes(const TcArgs &a);

// ---------------------------------------------------- skinny swap-AB path
struct SkinnyTcArgs {
    CUtensorMap tmB;   // B (N,K) bf16 K-major, box {64, 128}  (MMA operand "A")
    CUtensorMap tmA;   // A (M,K) bf16 K-major, box {64, MP}   (MMA operand "B")
    void *D;           // bf16 (M,N) row stride ldd
    int64_t ldd;
    int M, N, K;
    int mp;            // M rounded up to a multiple of 16, <= 64
    float *partials;   // scratch: grid * 2 slots of 128 * mp fp32
    uint32_t *counters;  // scratch: 4 per 128-row tile of B, zero on entry
    int grid;          // number of CTAs (persistent)
};
cudaError_t launch_skinny_tc(const SkinnyTcArgs &a, const ErrCtx &err, cudaStream_t s);
// The skinny kernel's fixed scratch in static device memory (for the entry
// point that allocates nothing).  First call per device looks up its device
// address with cudaGetSymbolAddress.
struct FixedScratch {
    float *partials;
    size_t partial_bytes;
    uint32_t *counters;
    size_t counter_bytes;
    int max_tiles;
};
cudaError_t skinny_fixed_scratch(FixedScratch *out);
// Scratch bytes the skinny path needs for a given problem and grid.
size_t skinny_partials_bytes(int grid, int mp);
size_t skinny_counters_bytes(int64_t N);

// ------------------------------------------------------------ MXFP4 path
struct Mxfp4Args {
    CUtensorMap tmA;    // A codes (M, K/2) u8, box {128, 128 (one CTA) | 128 (pair half)}, 128B swizzle
    CUtensorMap tmB;    // B codes (N, K/2) u8, box {128, 128 | bn/2}
    CUtensorMap tmSA;   // pair kernel: relaid A scales (wide form) as rows of 256 bytes, box {256, 16}
    CUtensorMap tmSB;   // pair kernel: relaid B scales (wide form), box {256, 16 * ceil(bn/128)}
    const uint8_t *sA;  // (M, K/32) e8m0
    const uint8_t *sB;  // (N, K/32) e8m0
    uint8_t *relA;      // scratch: sA relaid in the tensor core's chunk order
    uint8_t *relB;      // scratch: sB likewise
    void *D;            // bf16 (M,N) row-major, ldd = N
    int M, N, K;
    int bn;             // pair kernel tile width (192 or 128)
};
// One-CTA kernel (128 x 128 tiles).  Two launches: the scale relayout
// pre-pass, then the GEMM.
cudaError_t launch_mxfp4(const Mxfp4Args &a, int num_sms, const ErrCtx &err, cudaStream_t s);
// CTA-pair kernel (256 x bn tiles), also two launches.
cudaError_t launch_mxfp4_pair(const Mxfp4Args &a, int num_sms, const ErrCtx &err, cudaStream_t s);
int mxfp4_pair_pick_bn(int64_t M, int64_t N, int num_sms);
// Whether the pair kernel reads its scales in the wide (4x replicated) form.
bool mxfp4_pair_wide_scales();
// Relaid scale bytes for `rows` rows grouped by `group_rows`, compact or
// wide form (see mx_common.cuh).
size_t mxfp4_relaid_scale_bytes(int64_t rows, int64_t K, int group_rows, bool wide);
cudaError_t launch_mx_scale_relayout(const uint8_t *sA, int M, uint8_t *relA, int groupA, const uint8_t *sB,
                                     int N, uint8_t *relB, int groupB, int K, bool wide, int num_sms,
                                     cudaStream_t s);

// ------------------------------------------- general layouts -> tcgen05
// P (rows, ldp) dense bf16 = X read through layout L over (rows, cols),
// zero-padded for cols <= k < ldp.
cudaError_t launch_pack(const void *X, const DevLayout &L, int64_t rows, int64_t cols, void *P, int64_t ldp,
                        int num_sms, cudaStream_t s);
// D (through layout L over (rows, cols)) = S dense row-major bf16.
cudaError_t launch_unpack(const void *S, int64_t rows, int64_t cols, void *D, const DevLayout &L, int num_sms,
                          cudaStream_t s);

// Probe kernel for the bounded wait (never signalled barrier).
cudaError_t launch_wait_probe(const ErrCtx &err, cudaStream_t s);

// Counts every kernel launch made through the launchers above.
void note_launch();

// Raise a kernel's dynamic shared-memory limit once per device (cached).
cudaError_t ensure_smem_attr(const void *func, int bytes);

}  // namespace tmg
