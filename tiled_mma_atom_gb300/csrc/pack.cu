// pack.cu — the bridge from arbitrary layouts to the tensor-core kernels.
//
// pack:   P[r * ldp + k] = X[crd2idx((r, k), L)] for r < rows, k < cols, and
//         0 for cols <= k < ldp: a bf16 operand in any (Shape, Stride) layout
//         (MN-major, nested, strided, broadcast) becomes a dense K-major copy
//         whose rows the TMA tiles can read.
// unpack: D[crd2idx((r, c), L)] = S[r * cols + c]: a dense row-major result
//         scattered into an arbitrary output layout.
//
// Both move 64 x 64 tiles through shared memory so that the side addressed
// through the layout is read (or written) along whichever logical index is
// closer in memory, and the dense side along its contiguous rows: a
// transpose for MN-major data, a plain copy for K-major data.  HBM-bound:
// each element is read once and written once.
#include "layout.cuh"

namespace tmg {
namespace {

constexpr int kT = 64;
constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kPackThreads)
    pack_kernel(const uint16_t *__restrict__ X, DevLayout L, int64_t rows, int64_t cols,
                uint16_t *__restrict__ P, int64_t ldp, int src_row_fast)
{
    __shared__ uint16_t tile[kT][kT + 2];        // [row][k]; odd word pitch
    const int64_t tiles_k = (ldp + kT - 1) / kT;
    const int64_t tiles = (rows + kT - 1) / kT * tiles_k;
    for (int64_t id = blockIdx.x; id < tiles; id += gridDim.x) {
        const int64_t r0 = id / tiles_k * kT, k0 = id % tiles_k * kT;
        for (int i = threadIdx.x; i < kT * kT; i += kPackThreads) {
            const int a = i % kT, b = i / kT;    // a runs along the source's closer index
            const int rr = src_row_fast ? a : b, kk = src_row_fast ? b : a;
            const int64_t r = r0 + rr, k = k0 + kk;
            tile[rr][kk] = (r < rows && k < cols) ? X[crd2idx(L, r, k)] : static_cast<uint16_t>(0);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kT * kT; i += kPackThreads) {
            const int kk = i % kT, rr = i / kT;
            const int64_t r = r0 + rr, k = k0 + kk;
            if (r < rows && k < ldp)
                P[r * ldp + k] = tile[rr][kk];
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kPackThreads)
    unpack_kernel(const uint16_t *__restrict__ S, int64_t rows, int64_t cols, uint16_t *__restrict__ D,
                  DevLayout L, int dst_row_fast)
{
    __shared__ uint16_t tile[kT][kT + 2];        // [row][col]
    const int64_t tiles_c = (cols + kT - 1) / kT;
    const int64_t tiles = (rows + kT - 1) / kT * tiles_c;
    for (int64_t id = blockIdx.x; id < tiles; id += gridDim.x) {
        const int64_t r0 = id / tiles_c * kT, c0 = id % tiles_c * kT;
        for (int i = threadIdx.x; i < kT * kT; i += kPackThreads) {
            const int cc = i % kT, rr = i / kT;
            const int64_t r = r0 + rr, c = c0 + cc;
            if (r < rows && c < cols)
                tile[rr][cc] = S[r * cols + c];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kT * kT; i += kPackThreads) {
            const int a = i % kT, b = i / kT;
            const int rr = dst_row_fast ? a : b, cc = dst_row_fast ? b : a;
            const int64_t r = r0 + rr, c = c0 + cc;
            if (r < rows && c < cols)
                D[crd2idx(L, r, c)] = tile[rr][cc];
        }
        __syncthreads();
    }
}

// The common MN-major case — flat modes, unit row stride, columns ldk
// elements apart with 16-byte alignment: X(r, k) = X[r + k * ldk].  Both
// sides move 16 bytes per thread: a thread loads 8 consecutive rows of two
// adjacent columns k, k+1 and stores each row's pair (k, k+1) as one 32-bit
// word; 8 consecutive k of one row are then stored as one 16-byte vector.
// The tile is kept as 32-bit words, 33 per row: the transposed stores hit
// at most two words per bank and the row reads none.
__global__ void __launch_bounds__(kPackThreads)
    pack_mn_kernel(const uint16_t *__restrict__ X, int64_t ldk, int64_t rows, int64_t cols,
                   uint16_t *__restrict__ P, int64_t ldp)
{
    constexpr int kPitch = kT / 2 + 1;                        // words per tile row
    __shared__ uint32_t tile[kT * kPitch];                    // (row, k pair)
    const int64_t tiles_k = (ldp + kT - 1) / kT;
    const int64_t tiles = (rows + kT - 1) / kT * tiles_k;
    for (int64_t id = blockIdx.x; id < tiles; id += gridDim.x) {
        const int64_t r0 = id / tiles_k * kT, k0 = id % tiles_k * kT;
        for (int i = threadIdx.x; i < kT * kT / 16; i += kPackThreads) {
            const int rv = i % 8, kp = i / 8;                 // 8 row groups x 32 column pairs
            const int64_t r = r0 + rv * 8, k = k0 + 2 * kp;
            uint16_t h[2][8];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (k + c < cols && r + 7 < rows) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(X + r + (k + c) * ldk));
                    h[c][0] = v.x & 0xFFFF, h[c][1] = v.x >> 16, h[c][2] = v.y & 0xFFFF, h[c][3] = v.y >> 16;
                    h[c][4] = v.z & 0xFFFF, h[c][5] = v.z >> 16, h[c][6] = v.w & 0xFFFF, h[c][7] = v.w >> 16;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        h[c][e] = (k + c < cols && r + e < rows) ? X[r + e + (k + c) * ldk] : static_cast<uint16_t>(0);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                tile[(rv * 8 + e) * kPitch + kp] = static_cast<uint32_t>(h[0][e]) | static_cast<uint32_t>(h[1][e]) << 16;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kT * kT / 8; i += kPackThreads) {
            const int kv = i % 8, rr = i / 8;
            const int64_t r = r0 + rr, k = k0 + kv * 8;
            if (r < rows && k < ldp) {     // ldp is a multiple of 8: the whole vector is inside
                const uint32_t *w = &tile[rr * kPitch + kv * 4];
                *reinterpret_cast<uint4 *>(P + r * ldp + k) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        __syncthreads();
    }
}

int64_t abs64(int64_t v) { return v < 0 ? -v : v; }

// Whether consecutive rows sit closer in memory than consecutive columns.
int row_fast(const DevLayout &L) { return abs64(L.stride[0][0]) < abs64(L.stride[1][0]) ? 1 : 0; }

unsigned grid_for(int64_t tiles, int num_sms)
{
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    return static_cast<unsigned>(tiles < cap ? tiles : cap);
}

}  // namespace

cudaError_t launch_pack(const void *X, const DevLayout &L, int64_t rows, int64_t cols, void *P, int64_t ldp,
                        int num_sms, cudaStream_t s)
{
    const int64_t tiles = (rows + kT - 1) / kT * ((ldp + kT - 1) / kT);
    note_launch();
    const bool mn_fast = L.depth[0] == 1 && L.depth[1] == 1 && L.stride[0][0] == 1 && L.stride[1][0] > 0 &&
                         L.stride[1][0] % 8 == 0 && (reinterpret_cast<uintptr_t>(X) & 15u) == 0 && ldp % 8 == 0;
    if (mn_fast) {
        pack_mn_kernel<<<grid_for(tiles, num_sms), kPackThreads, 0, s>>>(
            static_cast<const uint16_t *>(X), L.stride[1][0], rows, cols, static_cast<uint16_t *>(P), ldp);
        return cudaGetLastError();
    }
    pack_kernel<<<grid_for(tiles, num_sms), kPackThreads, 0, s>>>(static_cast<const uint16_t *>(X), L, rows, cols,
                                                                   static_cast<uint16_t *>(P), ldp, row_fast(L));
    return cudaGetLastError();
}

cudaError_t launch_unpack(const void *S, int64_t rows, int64_t cols, void *D, const DevLayout &L, int num_sms,
                          cudaStream_t s)
{
    const int64_t tiles = (rows + kT - 1) / kT * ((cols + kT - 1) / kT);
    note_launch();
    unpack_kernel<<<grid_for(tiles, num_sms), kPackThreads, 0, s>>>(static_cast<const uint16_t *>(S), rows, cols,
                                                                     static_cast<uint16_t *>(D), L, row_fast(L));
    return cudaGetLastError();
}

}  // namespace tmg
