// tc2_bf16.cu — the bf16 GEMM on CTA pairs (kernel in tc2_kernel.cuh):
// the launches of the plain bf16 kernels, the schedule plan (data-parallel
// tiles and the stream-K tail) and the tile-width choice.
#include "tc2_kernel.cuh"

namespace tmg {

void tc2_plan(TcArgs &a, int num_sms)
{
    const int pairs = num_sms / 2;
    const int tiles = ((a.M + kBM - 1) / kBM) * ((a.N + a.bn - 1) / a.bn);
    const int kbe = a.kb_elems > 0 ? a.kb_elems : 64;
    const int num_kb = (a.K + kbe - 1) / kbe;
    const int full_waves = tiles / pairs;
    int dp = tiles, sk = 0;
    if (tiles % pairs != 0) {
        // the last full wave and the partial one run stream-K, provided
        // every pair gets at least one K block
        dp = (full_waves > 0 ? full_waves - 1 : 0) * pairs;
        sk = tiles - dp;
        if (static_cast<int64_t>(sk) * num_kb < pairs) {
            dp = tiles;
            sk = 0;
        }
    }
    a.dp_tiles = dp;
    a.sk_tiles = sk;
    a.pairs = sk > 0 ? pairs : (tiles < pairs ? tiles : pairs);
}

size_t tc2_partials_bytes(const TcArgs &a)
{
    return a.sk_tiles > 0 ? static_cast<size_t>(a.pairs) * 2 * kBM * a.bn * sizeof(float) : 0;
}

size_t tc2_counters_bytes(const TcArgs &a)
{
    // one counter per split tile, CTA and epilogue warp (up to 8 warps)
    return static_cast<size_t>(a.sk_tiles) * 2 * epi_warps(true) * sizeof(uint32_t);
}

int tc2_pick_bn(int64_t M, int64_t N, int num_sms)
{
    (void)M;
    (void)num_sms;
    // A pair MMA costs about the same at any width, so pick the width with
    // the least total cost over the column tiles: roughly (2000 + width) per
    // tile column (measured: 256-wide tiles do 14% more work than 224-wide
    // ones in the same time).
    static const int cands[] = {256, 224, 192, 128};
    int best = 256;
    int64_t best_cost = -1;
    for (int bn : cands) {
        const int64_t cost = ((N + bn - 1) / bn) * (2000 + bn);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

cudaError_t launch_tc2_bf16(const TcArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    (void)num_sms;
    const Tc2Epi none{nullptr, nullptr, nullptr, kEpiNone, 0};
    if (a.maj != 0) {
        // MN-major operands read in place (bn 256 or 128)
        const bool w = a.bn == 256;
        switch (a.maj) {
        case 1:
            return w ? launch_pair<256, kInBf16, false, 1>(a, none, err, s) : launch_pair<128, kInBf16, false, 1>(a, none, err, s);
        case 2:
            return w ? launch_pair<256, kInBf16, false, 2>(a, none, err, s) : launch_pair<128, kInBf16, false, 2>(a, none, err, s);
        default:
            return w ? launch_pair<256, kInBf16, false, 3>(a, none, err, s) : launch_pair<128, kInBf16, false, 3>(a, none, err, s);
        }
    }
    switch (a.bn) {
    case 256:
        return launch_pair<256, kInBf16, false>(a, none, err, s);
    case 224:
        return launch_pair<224, kInBf16, false>(a, none, err, s);
    case 192:
        return launch_pair<192, kInBf16, false>(a, none, err, s);
    default:
        return launch_pair<128, kInBf16, false>(a, none, err, s);
    }
}

}  // namespace tmg
