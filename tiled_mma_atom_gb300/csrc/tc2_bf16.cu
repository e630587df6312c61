// tc2_bf16.cu — the bf16 GEMM on CTA pairs (kernel in tc2_kernel.cuh):
// the launches of the plain bf16 kernels, the schedule plan (data-parallel
// tiles and the stream-K tail) and the tile-width choice.
#include <algorithm>
#include <cstdlib>

#include "tc2_kernel.cuh"

namespace tmg {

// Estimated time of the pair kernel in ns (up to a constant) for 256 x bn
// tiles over `pairs` CTA pairs, data-parallel (each pair takes whole tiles,
// the last wave possibly partial) or with a stream-K tail (the last full
// wave and the partial one split into equal runs of K blocks, summed from
// fp32 partials).  Per K block of one tile, measured on GB300 (bf16, L2
// flushed, sweep of M 2048-8192, N 1024-8192, K 2048-4096): 204 / 244 / 281
// / 320 ns at widths 128 / 192 / 224 / 256; a stream-K tail adds about 10 us
// (the partials' traffic and the ordered fix-up), so it pays only where a
// data-parallel last wave would leave many pairs idle for many K blocks.
static double tc2_kb_cost(int bn)
{
    return bn <= 128 ? 204.0 : bn <= 192 ? 244.0 : bn <= 224 ? 281.0 : 320.0;
}

static bool tc2_sk_possible(int64_t tiles, int num_kb, int pairs)
{
    if (tiles % pairs == 0)
        return false;
    const int64_t full_waves = tiles / pairs;
    const int64_t sk = tiles - (full_waves > 0 ? full_waves - 1 : 0) * pairs;
    return sk * num_kb >= pairs;
}

static double tc2_est(int64_t M, int64_t N, int num_kb, int bn, int pairs, bool sk)
{
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
    const double c = tc2_kb_cost(bn) * num_kb;
    if (sk && tc2_sk_possible(tiles, num_kb, pairs))
        return static_cast<double>(tiles) / pairs * c + 10000.0;
    return static_cast<double>((tiles + pairs - 1) / pairs) * c;
}

static int tc2_best_bn(int64_t M, int64_t N, int64_t K, int kb_elems, int num_sms, const int *cands, int nc,
                       double *est = nullptr)
{
    const int pairs = num_sms / 2;
    const int num_kb = static_cast<int>((K + kb_elems - 1) / kb_elems);
    int best = cands[0];
    double best_t = -1.0;
    for (int i = 0; i < nc; ++i) {
        const double t = std::min(tc2_est(M, N, num_kb, cands[i], pairs, false),
                                  tc2_est(M, N, num_kb, cands[i], pairs, true));
        if (best_t < 0.0 || t < best_t) {
            best_t = t;
            best = cands[i];
        }
    }
    if (est)
        *est = best_t;
    return best;
}

void tc2_plan(TcArgs &a, int num_sms)
{
    const int pairs = num_sms / 2;
    const int tiles = ((a.M + kBM - 1) / kBM) * ((a.N + a.bn - 1) / a.bn);
    const int kbe = a.kb_elems > 0 ? a.kb_elems : 64;
    const int num_kb = (a.K + kbe - 1) / kbe;
    bool sk = tc2_est(a.M, a.N, num_kb, a.bn, pairs, true) < tc2_est(a.M, a.N, num_kb, a.bn, pairs, false);
    if (const char *f = getenv("TMG_TC_PAIR_SCHED"))        // testing aid: "sk" | "dp"
        sk = f[0] == 's';
    int dp = tiles, skt = 0;
    if (sk && tc2_sk_possible(tiles, num_kb, pairs)) {
        // the last full wave and the partial one run stream-K
        const int full_waves = tiles / pairs;
        dp = (full_waves > 0 ? full_waves - 1 : 0) * pairs;
        skt = tiles - dp;
    }
    a.dp_tiles = dp;
    a.sk_tiles = skt;
    // Tile groups of 16 M-tiles when their A panels (16 x 256 rows x K)
    // take at most 32 MB, a quarter of L2: at bf16 4096^3 a wave of 76 pairs
    // then covers all 16 M-tiles and five columns of B, every A panel stays
    // in L2 across the waves, and DRAM reads fall from 1.27x the operands
    // (groups of 8) to 1.08x (ncu); the fp8 8192^3 GEMM reads 303 MB per
    // launch instead of 389 MB.  With larger panels (bf16 K = 8192: 64 MB)
    // the group no longer stays in L2 beside the B columns and groups of 8
    // read less (1.23 GB against 1.54 GB per launch at 8192^3).
    const int64_t panel_bytes = static_cast<int64_t>(kBM) * num_kb * kbe * (kbe == 128 ? 1 : 2);
    a.group_m = 16 * panel_bytes <= (int64_t{32} << 20) ? 16 : 8;
    a.pairs = skt > 0 ? pairs : (tiles < pairs ? tiles : pairs);
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

int tc2_pick_bn(int64_t M, int64_t N, int64_t K, int num_sms, double *est_ns)
{
    static const int cands[] = {256, 224, 192, 128};
    return tc2_best_bn(M, N, K, 64, num_sms, cands, 4, est_ns);
}

int tc2_pick_bn_of(int64_t M, int64_t N, int64_t K, int kb_elems, int num_sms, const int *cands, int nc)
{
    return tc2_best_bn(M, N, K, kb_elems, num_sms, cands, nc);
}

cudaError_t launch_tc2_bf16(const TcArgs &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    (void)num_sms;
    const Tc2Epi none{nullptr, nullptr, nullptr, kEpiNone, 0};
    if (a.maj == 1) {
        // MN-major A read in place (any width: its boxes do not depend on it)
        switch (a.bn) {
        case 256:
            return launch_pair<256, kInBf16, false, 1>(a, none, err, s);
        case 224:
            return launch_pair<224, kInBf16, false, 1>(a, none, err, s);
        case 192:
            return launch_pair<192, kInBf16, false, 1>(a, none, err, s);
        case 128:
            return launch_pair<128, kInBf16, false, 1>(a, none, err, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    if (a.maj != 0) {
        // MN-major B read in place: 64-column boxes, so bn 256 or 128
        if (a.bn != 256 && a.bn != 128)
            return cudaErrorInvalidValue;
        const bool w = a.bn == 256;
        switch (a.maj) {
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
    case 128:
        return launch_pair<128, kInBf16, false>(a, none, err, s);
    default:
        return cudaErrorInvalidValue;     // a width no kernel is built for
    }
}

}  // namespace tmg
