// api.cu — the library's C ABI (include/tmg.h): argument validation, layout
// classification, TMA descriptor encoding, kernel-family dispatch and error
// reporting.
//
// Layout handling follows "FlyDSL Kernel Authoring Skill", §2 "Layout
// System": a layout is a (Shape, Stride) pair and element (i,j) sits at
// crd2idx((i,j)) = Σ coordinate × stride.  The host classifies each operand
// layout:
//   K-major dense   (rows, K):(ld, 1)  -> TMA tiles, tcgen05 K-major operand
//   anything else (MN-major, nested, strided, broadcast) -> for problems
//                   large enough to pay for it, a crd2idx gather into a
//                   K-major scratch copy (pack.cu) and then the tensor
//                   cores; else the CUDA-core path, which evaluates
//                   crd2idx per element.
// D given column-major, (M,N):(1,ld), is computed as Dᵀ = B·Aᵀ with the
// operand roles swapped, so it also reaches the tensor-core kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <unordered_map>
#include <mutex>
#include <string>
#include <utility>

#include "internal.h"
#include "tmg.h"

namespace tmg {

__device__ uint32_t g_err_word;

namespace {

thread_local std::string t_last_error;
std::atomic<uint64_t> g_budget_ns{2000000000ull};
std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *err_word = nullptr;
};
std::map<int, DeviceState> g_dev;

struct Scratch {
    float *partials = nullptr;
    size_t partials_bytes = 0;
    uint32_t *counters = nullptr;
    size_t counters_bytes = 0;
    uint8_t *mx_scales = nullptr;      // MXFP4 scales in chunk order
    size_t mx_scales_bytes = 0;
    float *tc2_partials = nullptr;     // pair kernel stream-K partial tiles
    size_t tc2_partials_bytes = 0;
    uint32_t *tc2_counters = nullptr;  // pair kernel stream-K tile counters
    size_t tc2_counters_bytes = 0;
    void *pack[3] = {nullptr, nullptr, nullptr};   // packed A, packed B, dense D
    size_t pack_bytes[3] = {0, 0, 0};
    void *host_ws[3] = {nullptr, nullptr, nullptr};  // tmg_gemm_host: device A, B, D
    size_t host_ws_bytes[3] = {0, 0, 0};
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    static constexpr int kHostEvents = 2 + 3 * 16;
    cudaEvent_t ev[kHostEvents] = {};
};
std::map<std::pair<int, uintptr_t>, Scratch> g_scratch;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// TMG_LOG=1 (any value but "0"): one line on stderr per GEMM call naming the
// kernel family, tile and schedule the dispatch chose.
bool log_on()
{
    static const bool on = [] {
        const char *v = getenv("TMG_LOG");
        return v && *v && strcmp(v, "0") != 0;
    }();
    return on;
}

void log_choice(const char *fmt, ...) __attribute__((format(printf, 1, 2)));
void log_choice(const char *fmt, ...)
{
    if (!log_on())
        return;
    char buf[400];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    fprintf(stderr, "tmg: %s\n", buf);
}

tmg_status fail(tmg_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
tmg_status fail(tmg_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

tmg_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(TMG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Per-device set-up, with that device current.
tmg_status device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &ds = g_dev[dev];
    if (!ds.ready) {
        if ((e = cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        cudaDeviceGetAttribute(&ds.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&ds.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (ds.cc_major != 10 || ds.cc_minor != 3)
            return fail(TMG_ERR_UNSUPPORTED,
                        "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev,
                        ds.cc_major, ds.cc_minor);
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_err_word)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        ds.err_word = static_cast<uint32_t *>(p);
        if ((e = cudaMemset(ds.err_word, 0, sizeof(uint32_t))) != cudaSuccess)
            return cuda_fail(e, "cudaMemset(error word)");
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail(TMG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        ds.ready = true;
    }
    *out = &ds;
    return TMG_OK;
}

ErrCtx err_ctx(const DeviceState &ds)
{
    return ErrCtx{ds.err_word, g_budget_ns.load()};
}

// ------------------------------------------------------------- layouts

int64_t mode_size(const tmg_layout &L, int t)
{
    return L.depth[t] == 2 ? L.shape[t][0] * L.shape[t][1] : L.shape[t][0];
}

tmg_layout row_major(int64_t rows, int64_t cols)
{
    tmg_layout L;
    std::memset(&L, 0, sizeof L);
    L.depth[0] = L.depth[1] = 1;
    L.shape[0][0] = rows;
    L.shape[1][0] = cols;
    L.stride[0][0] = cols;
    L.stride[1][0] = 1;
    L.shape[0][1] = L.shape[1][1] = 1;
    return L;
}

// Checks depth, shapes and extents; strides >= 0 (> 0 when `output`);
// the largest offset must fit in int64.
tmg_status check_layout(const tmg_layout &L, int64_t rows, int64_t cols, bool output, const char *name)
{
    const int64_t ext[2] = {rows, cols};
    __int128 max_off = 0;
    for (int t = 0; t < 2; ++t) {
        if (L.depth[t] != 1 && L.depth[t] != 2)
            return fail(TMG_ERR_INVALID_ARG, "%s: mode %d depth %d (must be 1 or 2)", name, t, L.depth[t]);
        for (int j = 0; j < L.depth[t]; ++j) {
            if (L.shape[t][j] < 1)
                return fail(TMG_ERR_INVALID_ARG, "%s: mode %d shape %lld < 1", name, t, (long long)L.shape[t][j]);
            if (L.stride[t][j] < 0 || (output && L.stride[t][j] == 0 && L.shape[t][j] > 1))
                return fail(TMG_ERR_INVALID_ARG, "%s: mode %d stride %lld not allowed", name, t,
                            (long long)L.stride[t][j]);
            max_off += static_cast<__int128>(L.shape[t][j] - 1) * L.stride[t][j];
        }
        if (mode_size(L, t) != ext[t])
            return fail(TMG_ERR_INVALID_ARG, "%s: mode %d has size %lld, expected %lld", name, t,
                        (long long)mode_size(L, t), (long long)ext[t]);
    }
    if (max_off > static_cast<__int128>(INT64_MAX / 2))
        return fail(TMG_ERR_INVALID_ARG, "%s: offsets overflow int64", name);
    return TMG_OK;
}

// Returns the row stride if L is (rows, cols):(ld, 1) with flat modes, else -1.
int64_t row_stride_if_rowmajor(const tmg_layout &L, int64_t rows, int64_t cols)
{
    if (L.depth[0] != 1 || L.depth[1] != 1)
        return -1;
    if (cols > 1 && L.stride[1][0] != 1)
        return -1;
    if (rows == 1)
        return L.stride[0][0] > 0 ? L.stride[0][0] : cols;
    return L.stride[0][0] > 0 ? L.stride[0][0] : -1;
}

// Column stride if L is (rows, cols):(1, ld) with flat modes, else -1.
int64_t col_stride_if_colmajor(const tmg_layout &L, int64_t rows, int64_t cols)
{
    if (L.depth[0] != 1 || L.depth[1] != 1)
        return -1;
    if (rows > 1 && L.stride[0][0] != 1)
        return -1;
    if (cols == 1)
        return L.stride[1][0] > 0 ? L.stride[1][0] : rows;
    return L.stride[1][0] > 0 ? L.stride[1][0] : -1;
}

DevLayout to_dev(const tmg_layout &L)
{
    DevLayout d;
    std::memcpy(&d, &L, sizeof d);
    static_assert(sizeof(DevLayout) == sizeof(tmg_layout), "layout struct mismatch");
    return d;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D TMA descriptor over a row-major (rows, inner) matrix of `elem` bytes
// with row stride `ld` elements: box {box_inner, box_rows}, 128-byte swizzle,
// out-of-range elements read as zero.
// Encoded descriptors are cached: a descriptor only records an address,
// extents, strides and the box, so an identical request gets an identical
// descriptor whatever the memory holds now.
struct MapKey {
    uintptr_t base;
    int64_t inner, rows, ld;
    int box_inner, box_rows, dt, swizzle;
    bool operator==(const MapKey &o) const
    {
        return base == o.base && inner == o.inner && rows == o.rows && ld == o.ld && box_inner == o.box_inner &&
               box_rows == o.box_rows && dt == o.dt && swizzle == o.swizzle;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const
    {
        uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
        for (uint64_t v : {static_cast<uint64_t>(k.inner), static_cast<uint64_t>(k.rows), static_cast<uint64_t>(k.ld),
                           static_cast<uint64_t>(k.box_inner) << 32 | static_cast<uint32_t>(k.box_rows),
                           static_cast<uint64_t>(k.dt) << 32 | static_cast<uint32_t>(k.swizzle)})
            h = (h ^ v) * 0x100000001B3ull;
        return static_cast<size_t>(h);
    }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
constexpr size_t kMaxCachedMaps = 1024;

tmg_status encode_2d(CUtensorMap *map, CUtensorMapDataType dt, int elem, const void *base,
                     int64_t inner, int64_t rows, int64_t ld, int box_inner, int box_rows,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    const MapKey key{reinterpret_cast<uintptr_t>(base), inner, rows, ld, box_inner, box_rows, static_cast<int>(dt),
                     static_cast<int>(swizzle)};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *map = it->second;
            return TMG_OK;
        }
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * elem};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TMG_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled failed (%d) for %lldx%lld ld=%lld", (int)r,
                    (long long)rows, (long long)inner, (long long)ld);
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() >= kMaxCachedMaps)
        g_maps.clear();
    g_maps.emplace(key, *map);
    return TMG_OK;
}

// TMA limits: 16-byte aligned base, row stride a multiple of 16 bytes and
// below 2^40, dimensions below 2^31 (kernel coordinates are int32).
bool tma_ok(const void *p, int64_t ld, int elem, int64_t rows, int64_t inner)
{
    return aligned16(p) && (ld * elem) % 16 == 0 && ld * elem < (int64_t(1) << 40) && rows < (int64_t(1) << 31) &&
           inner < (int64_t(1) << 31) && ld >= 1;
}

// Tensor-core plan: operands after a possible swap, all K-major.
struct TcPlan {
    bool ok = false;
    const void *A, *B;
    int64_t M, N, lda, ldb, ldd;
};

TcPlan plan_tc(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, const tmg_layout &la,
               const tmg_layout &lb, const tmg_layout &ld)
{
    TcPlan p;
    const int64_t lda = row_stride_if_rowmajor(la, M, K);
    const int64_t ldb = row_stride_if_rowmajor(lb, N, K);
    if (lda < 0 || ldb < 0)
        return p;
    int64_t ldd = row_stride_if_rowmajor(ld, M, N);
    if (ldd > 0 && (N == 1 || ldd >= N)) {
        p = TcPlan{true, A, B, M, N, lda, ldb, ldd};
    } else {
        ldd = col_stride_if_colmajor(ld, M, N);
        if (ldd > 0 && (M == 1 || ldd >= M))
            p = TcPlan{true, B, A, N, M, ldb, lda, ldd};
    }
    if (!p.ok)
        return p;
    if (!tma_ok(p.A, p.lda, 2, p.M, K) || !tma_ok(p.B, p.ldb, 2, p.N, K) || p.M > INT32_MAX ||
        p.N > INT32_MAX || K > INT32_MAX)
        p.ok = false;
    (void)D;
    return p;
}

Scratch *skinny_scratch(int dev, cudaStream_t s, size_t pbytes, size_t cbytes, tmg_status *st)
{
    std::lock_guard<std::mutex> lk(g_mu);
    Scratch &sc = g_scratch[{dev, reinterpret_cast<uintptr_t>(s)}];
    cudaError_t e;
    if (sc.partials_bytes < pbytes) {
        if (sc.partials)
            cudaFree(sc.partials);
        sc.partials = nullptr;
        sc.partials_bytes = 0;
        if ((e = cudaMalloc(&sc.partials, pbytes)) != cudaSuccess) {
            *st = cuda_fail(e, "cudaMalloc(skinny partials)");
            return nullptr;
        }
        sc.partials_bytes = pbytes;
    }
    if (sc.counters_bytes < cbytes) {
        if (sc.counters)
            cudaFree(sc.counters);
        sc.counters = nullptr;
        sc.counters_bytes = 0;
        if ((e = cudaMalloc(&sc.counters, cbytes)) != cudaSuccess) {
            *st = cuda_fail(e, "cudaMalloc(skinny counters)");
            return nullptr;
        }
        if ((e = cudaMemsetAsync(sc.counters, 0, cbytes, s)) != cudaSuccess) {
            *st = cuda_fail(e, "cudaMemsetAsync(skinny counters)");
            return nullptr;
        }
        sc.counters_bytes = cbytes;
    }
    *st = TMG_OK;
    return &sc;
}

// Per-(device, stream) buffer for the MXFP4 scale relayout, grown on demand.
uint8_t *mx_scale_scratch(int dev, cudaStream_t s, size_t bytes, tmg_status *st)
{
    std::lock_guard<std::mutex> lk(g_mu);
    Scratch &sc = g_scratch[{dev, reinterpret_cast<uintptr_t>(s)}];
    if (sc.mx_scales_bytes < bytes) {
        if (sc.mx_scales)
            cudaFree(sc.mx_scales);
        sc.mx_scales = nullptr;
        sc.mx_scales_bytes = 0;
        cudaError_t e = cudaMalloc(&sc.mx_scales, bytes);
        if (e != cudaSuccess) {
            *st = cuda_fail(e, "cudaMalloc(MXFP4 scale relayout)");
            return nullptr;
        }
        sc.mx_scales_bytes = bytes;
    }
    *st = TMG_OK;
    return sc.mx_scales;
}

// mode: 0 = choose, 1 = one-CTA tiles, 2 = CTA-pair tiles.
// Per-(device, stream) stream-K scratch of the pair kernel, grown on demand;
// counters are zeroed when allocated and reset by the kernel after use.
tmg_status tc2_scratch(int dev, cudaStream_t s, TcArgs &a)
{
    const size_t pb = tc2_partials_bytes(a), cb = tc2_counters_bytes(a);
    a.partials = nullptr;
    a.counters = nullptr;
    if (pb == 0)
        return TMG_OK;
    std::lock_guard<std::mutex> lk(g_mu);
    Scratch &sc = g_scratch[{dev, reinterpret_cast<uintptr_t>(s)}];
    cudaError_t e;
    if (sc.tc2_partials_bytes < pb) {
        if (sc.tc2_partials)
            cudaFree(sc.tc2_partials);
        sc.tc2_partials = nullptr;
        sc.tc2_partials_bytes = 0;
        if ((e = cudaMalloc(&sc.tc2_partials, pb)) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(pair stream-K partials)");
        sc.tc2_partials_bytes = pb;
    }
    if (sc.tc2_counters_bytes < cb) {
        if (sc.tc2_counters)
            cudaFree(sc.tc2_counters);
        sc.tc2_counters = nullptr;
        sc.tc2_counters_bytes = 0;
        if ((e = cudaMalloc(&sc.tc2_counters, cb)) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(pair stream-K counters)");
        if ((e = cudaMemsetAsync(sc.tc2_counters, 0, cb, s)) != cudaSuccess)
            return cuda_fail(e, "cudaMemsetAsync(pair stream-K counters)");
        sc.tc2_counters_bytes = cb;
    }
    a.partials = sc.tc2_partials;
    a.counters = sc.tc2_counters;
    return TMG_OK;
}

// Testing aid: TMG_TC_PAIR_BN = 128 | 192 | 224 | 256 forces the pair-tile
// width of the plain and fused pair kernels.
int pair_bn_override(int bn)
{
    if (const char *f = getenv("TMG_TC_PAIR_BN")) {
        const int v = atoi(f);
        if (v == 128 || v == 192 || v == 224 || v == 256)
            return v;
    }
    return bn;
}

tmg_status run_tc(const DeviceState &ds, const TcPlan &p, void *D, int64_t K, int mode, cudaStream_t s)
{
    TcArgs a;
    std::memset(&a, 0, sizeof a);
    // CTA pairs or one-CTA tiles, whichever the cost model expects to be
    // faster: pairs halve the B traffic per SM, one-CTA tiles come in twice
    // as many per wave.
    bool pair = mode == 2;
    double est1 = 0.0, est2 = 0.0;
    const int bn1 = tc_pick_bn(p.M, p.N, K, ds.num_sms, &est1);
    if (mode == 0 && p.M >= 256) {
        tc2_pick_bn(p.M, p.N, K, ds.num_sms, &est2);
        pair = est2 < est1;
    }
    int box_b;
    if (pair) {
        a.bn = pair_bn_override(tc2_pick_bn(p.M, p.N, K, ds.num_sms));
        box_b = a.bn / 2;
    } else {
        a.bn = bn1;
        box_b = a.bn;
    }
    tmg_status st;
    if ((st = encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.A, K, p.M, p.lda, 64, 128)) != TMG_OK)
        return st;
    if ((st = encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.B, K, p.N, p.ldb, 64, box_b)) != TMG_OK)
        return st;
    a.D = D;
    a.ldd = p.ldd;
    a.M = static_cast<int>(p.M);
    a.N = static_cast<int>(p.N);
    a.K = static_cast<int>(K);
    if (pair) {
        tc2_plan(a, ds.num_sms);
        int dev = 0;
        cudaGetDevice(&dev);
        if ((st = tc2_scratch(dev, s, a)) != TMG_OK)
            return st;
    }
    if (pair)
        log_choice("bf16 %dx%dx%d -> tc2_gemm_kernel (CTA pairs): 256x%d tiles, %d pairs, %d data-parallel + %d "
                   "stream-K tiles, groups of %d M-tiles", a.M, a.N, a.K, a.bn, a.pairs, a.dp_tiles, a.sk_tiles, a.group_m);
    else
        log_choice("bf16 %dx%dx%d -> tc_bf16_kernel (one CTA): 128x%d tiles", a.M, a.N, a.K, a.bn);
    cudaError_t e = pair ? launch_tc2_bf16(a, ds.num_sms, err_ctx(ds), s) : launch_tc_bf16(a, ds.num_sms, err_ctx(ds), s);
    return e == cudaSuccess ? TMG_OK : cuda_fail(e, pair ? "tc2_bf16 launch" : "tc_bf16 launch");
}

// Per-(device, stream) buffer `which` (0: packed A, 1: packed B, 2: dense D)
// of the general-layout path, grown on demand.
void *pack_scratch(int which, size_t bytes, cudaStream_t s, tmg_status *st)
{
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_mu);
    Scratch &sc = g_scratch[{dev, reinterpret_cast<uintptr_t>(s)}];
    if (sc.pack_bytes[which] < bytes) {
        if (sc.pack[which])
            cudaFree(sc.pack[which]);
        sc.pack[which] = nullptr;
        sc.pack_bytes[which] = 0;
        cudaError_t e = cudaMalloc(&sc.pack[which], bytes);
        if (e != cudaSuccess) {
            *st = cuda_fail(e, "cudaMalloc(general-layout workspace)");
            return nullptr;
        }
        sc.pack_bytes[which] = bytes;
    }
    *st = TMG_OK;
    return sc.pack[which];
}

tmg_status run_skinny(const DeviceState &ds, const TcPlan &p, void *D, int64_t K, cudaStream_t s);

// Device workspace and copy streams of tmg_gemm_host for (device, stream).
Scratch *host_scratch(cudaStream_t s, const size_t (&bytes)[3], tmg_status *st)
{
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_mu);
    Scratch &sc = g_scratch[{dev, reinterpret_cast<uintptr_t>(s)}];
    cudaError_t e;
    if (!sc.copy_in) {
        if ((e = cudaStreamCreateWithFlags(&sc.copy_in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&sc.copy_out, cudaStreamNonBlocking)) != cudaSuccess) {
            *st = cuda_fail(e, "cudaStreamCreate(host copy streams)");
            return nullptr;
        }
        for (cudaEvent_t &ev : sc.ev)
            if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) {
                *st = cuda_fail(e, "cudaEventCreate(host copy events)");
                return nullptr;
            }
    }
    for (int i = 0; i < 3; ++i) {
        if (sc.host_ws_bytes[i] >= bytes[i])
            continue;
        if (sc.host_ws[i])
            cudaFree(sc.host_ws[i]);
        sc.host_ws[i] = nullptr;
        sc.host_ws_bytes[i] = 0;
        if ((e = cudaMalloc(&sc.host_ws[i], bytes[i])) != cudaSuccess) {
            *st = cuda_fail(e, "cudaMalloc(host-buffer GEMM workspace)");
            return nullptr;
        }
        sc.host_ws_bytes[i] = bytes[i];
    }
    *st = TMG_OK;
    return &sc;
}

// Operands given MN-major (M or N contiguous: (rows, K):(1, ld)) read in
// place by the pair kernel, together with K-major ones, when the problem is
// large enough for CTA pairs and D is row-major.  Returns false when it does
// not apply (the caller gathers instead).
bool run_tc2_inplace(const DeviceState &ds, const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                     const tmg_layout &la, const tmg_layout &lb, const tmg_layout &ld, cudaStream_t s,
                     tmg_status *st)
{
    const int64_t ldd = row_stride_if_rowmajor(ld, M, N);
    if (ldd <= 0 || (N > 1 && ldd < N) || M < 256 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return false;
    const void *ops[2] = {A, B};
    const tmg_layout *lays[2] = {&la, &lb};
    const int64_t rows[2] = {M, N};
    int64_t lds[2];
    int maj = 0;
    for (int i = 0; i < 2; ++i) {
        lds[i] = row_stride_if_rowmajor(*lays[i], rows[i], K);
        if (lds[i] > 0 && tma_ok(ops[i], lds[i], 2, rows[i], K))
            continue;
        lds[i] = col_stride_if_colmajor(*lays[i], rows[i], K);
        if (lds[i] > 0 && lds[i] >= rows[i] && tma_ok(ops[i], lds[i], 2, K, rows[i])) {
            maj |= 1 << i;
            continue;
        }
        return false;
    }
    if (maj == 0)
        return false;                                     // the ordinary dispatch covers it
    TcArgs a;
    std::memset(&a, 0, sizeof a);
    a.maj = maj;
    // an MN-major B is read in 64-column boxes: widths 256 and 128 only
    static const int kBMnWidths[2] = {256, 128};
    if (maj & 2) {
        a.bn = tc2_pick_bn_of(M, N, K, 64, ds.num_sms, kBMnWidths, 2);
        const int f = pair_bn_override(a.bn);
        a.bn = (f == 256 || f == 128) ? f : a.bn;
    } else {
        a.bn = pair_bn_override(tc2_pick_bn(M, N, K, ds.num_sms));
    }
    if (((M + 255) / 256) * ((N + a.bn - 1) / a.bn) < ds.num_sms / 2)
        return false;                                     // too few pair tiles
    if ((*st = (maj & 1) ? encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, M, K, lds[0], 64, 64)
                         : encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, lds[0], 64, 128)) != TMG_OK)
        return true;
    if ((*st = (maj & 2) ? encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, N, K, lds[1], 64, 64)
                         : encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, K, N, lds[1], 64, a.bn / 2)) !=
        TMG_OK)
        return true;
    a.D = D;
    a.ldd = ldd;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    tc2_plan(a, ds.num_sms);
    int dev = 0;
    cudaGetDevice(&dev);
    if ((*st = tc2_scratch(dev, s, a)) != TMG_OK)
        return true;
    log_choice("bf16 %dx%dx%d -> tc2_gemm_kernel (CTA pairs), MN-major operands read in place (A %s, B %s): "
               "256x%d tiles, %d pairs, %d data-parallel + %d stream-K tiles, groups of %d M-tiles", a.M, a.N, a.K,
               (a.maj & 1) ? "MN-major" : "K-major", (a.maj & 2) ? "MN-major" : "K-major", a.bn, a.pairs, a.dp_tiles,
               a.sk_tiles, a.group_m);
    const cudaError_t e = launch_tc2_bf16(a, ds.num_sms, err_ctx(ds), s);
    *st = e == cudaSuccess ? TMG_OK : cuda_fail(e, "tc2_bf16 (MN-major operands) launch");
    return true;
}

// General layouts on the tensor cores: every operand the TMA cannot read in
// place is gathered through its layout into a dense K-major scratch copy
// (rows padded to a multiple of 8 elements), a D that is neither row- nor
// column-major gets a dense row-major scratch result that is scattered back
// through its layout; the GEMM in between is the ordinary tcgen05 dispatch.
tmg_status run_packed(const DeviceState &ds, const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                      const tmg_layout &la, const tmg_layout &lb, const tmg_layout &ld, cudaStream_t s)
{
    tmg_status st;
    cudaError_t e;
    if (!getenv("TMG_NO_INPLACE_MN") && run_tc2_inplace(ds, A, B, D, M, N, K, la, lb, ld, s, &st))
        return st;
    const int64_t Kp = (K + 7) / 8 * 8;
    const void *ops[2] = {A, B};
    const tmg_layout *lays[2] = {&la, &lb};
    const int64_t rows[2] = {M, N};
    int64_t lds[2];
    for (int i = 0; i < 2; ++i) {
        lds[i] = row_stride_if_rowmajor(*lays[i], rows[i], K);
        if (lds[i] > 0 && tma_ok(ops[i], lds[i], 2, rows[i], K))
            continue;
        void *P = pack_scratch(i, static_cast<size_t>(rows[i]) * Kp * 2, s, &st);
        if (!P)
            return st;
        if ((e = launch_pack(ops[i], to_dev(*lays[i]), rows[i], K, P, Kp, ds.num_sms, s)) != cudaSuccess)
            return cuda_fail(e, "pack launch");
        ops[i] = P;
        lds[i] = Kp;
    }
    tmg_layout pa = row_major(M, K), pb = row_major(N, K);
    pa.stride[0][0] = lds[0];
    pb.stride[0][0] = lds[1];
    TcPlan p = plan_tc(ops[0], ops[1], D, M, N, K, pa, pb, ld);
    void *dense = nullptr;
    if (!p.ok) {
        dense = pack_scratch(2, static_cast<size_t>(M) * N * 2, s, &st);
        if (!dense)
            return st;
        p = plan_tc(ops[0], ops[1], dense, M, N, K, pa, pb, row_major(M, N));
        if (!p.ok)
            return fail(TMG_ERR_UNSUPPORTED, "general-layout path: extents beyond the tensor-core kernels' limits");
    }
    void *Dout = dense ? dense : D;
    st = p.M <= 64 ? run_skinny(ds, p, Dout, K, s) : run_tc(ds, p, Dout, K, 0, s);
    if (st != TMG_OK || !dense)
        return st;
    if ((e = launch_unpack(dense, M, N, D, to_dev(ld), ds.num_sms, s)) != cudaSuccess)
        return cuda_fail(e, "unpack launch");
    return TMG_OK;
}

tmg_status run_skinny(const DeviceState &ds, const TcPlan &p, void *D, int64_t K, cudaStream_t s)
{
    SkinnyTcArgs a;
    std::memset(&a, 0, sizeof a);
    a.mp = static_cast<int>((p.M + 15) / 16 * 16);
    tmg_status st;
    if ((st = encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.B, K, p.N, p.ldb, 64, 128)) != TMG_OK)
        return st;
    if ((st = encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.A, K, p.M, p.lda, 64, a.mp)) != TMG_OK)
        return st;
    const int64_t units = ((p.N + 127) / 128) * ((K + 63) / 64);
    a.grid = static_cast<int>(units < ds.num_sms ? units : ds.num_sms);
    int dev = 0;
    cudaGetDevice(&dev);
    Scratch *sc = skinny_scratch(dev, s, skinny_partials_bytes(a.grid, a.mp), skinny_counters_bytes(p.N), &st);
    if (!sc)
        return st;
    a.partials = sc->partials;
    a.counters = sc->counters;
    a.D = D;
    a.ldd = p.ldd;
    a.M = static_cast<int>(p.M);
    a.N = static_cast<int>(p.N);
    a.K = static_cast<int>(K);
    log_choice("bf16 %dx%dx%d -> skinny_tc_kernel (swap-AB, MMA N = %d): stream-K over %lld units on %d CTAs", a.M,
               a.N, a.K, a.mp, static_cast<long long>(units), a.grid);
    cudaError_t e = launch_skinny_tc(a, err_ctx(ds), s);
    return e == cudaSuccess ? TMG_OK : cuda_fail(e, "skinny_tc launch");
}

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

cudaError_t ensure_smem_attr(const void *func, int bytes)
{
    // The attribute is an upper bound on the dynamic shared memory of later
    // launches, so it only ever grows: remember the largest value set per
    // (device, kernel) — kernels whose size depends on the problem launch
    // with several sizes.
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> largest;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const auto key = std::make_pair(dev, func);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = largest.find(key);
        if (it != largest.end() && it->second >= bytes)
            return cudaSuccess;
    }
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lk(mu);
        int &v = largest[key];
        if (v < bytes)
            v = bytes;
    }
    return e;
}

namespace {

__global__ void wait_probe_kernel(ErrCtx err)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait(&bar, 0, err, nullptr, kSiteProbe);   // nothing ever arrives
}

#ifdef TMG_DEBUG_BOUNDS
// Checks the offset `limit` against a buffer of `limit` elements — one past
// its end — and touches no memory either way: the debug build's check must
// record it in the device error word.
__global__ void bounds_probe_kernel(int64_t limit, ErrCtx err)
{
    if (threadIdx.x == 0)
        (void)bounds_ok(limit, limit, err, kBndProbe);
}
#endif

}  // namespace

cudaError_t launch_wait_probe(const ErrCtx &err, cudaStream_t s)
{
    note_launch();
    wait_probe_kernel<<<1, 32, 0, s>>>(err);
    return cudaGetLastError();
}

}  // namespace tmg

using namespace tmg;

extern "C" {

tmg_status tmg_gemm_ex(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                       tmg_dtype dtype, const tmg_layout *layoutA, const tmg_layout *layoutB,
                       const tmg_layout *layoutD, tmg_path path, void *stream)
{
    t_last_error.clear();
    if (dtype == TMG_E4M3)
        return fail(TMG_ERR_INVALID_ARG, "E4M3 is an input type of tmg_gemm_fused only (D is bf16 there)");
    if (dtype != TMG_F32 && dtype != TMG_BF16)
        return fail(TMG_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (path < TMG_PATH_AUTO || path > TMG_PATH_PACKED_TC)
        return fail(TMG_ERR_INVALID_ARG, "unknown path %d", (int)path);
    if (M < 0 || N < 0 || K < 0)
        return fail(TMG_ERR_INVALID_ARG, "negative extent M=%lld N=%lld K=%lld", (long long)M, (long long)N,
                    (long long)K);
    if (M == 0 || N == 0)
        return TMG_OK;
    if (!D || (K > 0 && (!A || !B)))
        return fail(TMG_ERR_INVALID_ARG, "null operand pointer");
    const tmg_layout la = layoutA ? *layoutA : row_major(M, K);
    const tmg_layout lb = layoutB ? *layoutB : row_major(N, K);
    const tmg_layout ld = layoutD ? *layoutD : row_major(M, N);
    tmg_status st;
    if (K > 0) {
        if ((st = check_layout(la, M, K, false, "layoutA")) != TMG_OK)
            return st;
        if ((st = check_layout(lb, N, K, false, "layoutB")) != TMG_OK)
            return st;
    }
    if ((st = check_layout(ld, M, N, true, "layoutD")) != TMG_OK)
        return st;

    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int dt = dtype == TMG_F32 ? 0 : 1;

    if (K == 0) {
        cudaError_t e = launch_zero_fill(D, to_dev(ld), M, N, dt, s);
        return e == cudaSuccess ? TMG_OK : cuda_fail(e, "zero_fill launch");
    }

    tmg_path use = path;
    TcPlan plan;
    if (dtype == TMG_BF16)
        plan = plan_tc(A, B, D, M, N, K, la, lb, ld);
    if (use == TMG_PATH_AUTO) {
        if (dtype == TMG_F32)
            use = TMG_PATH_FFMA;
        else if (!plan.ok)
            // the gather pays for itself once the product is at least 512³
            use = static_cast<double>(M) * N * K >= 134217728.0 ? TMG_PATH_PACKED_TC : TMG_PATH_FFMA;
        else
            use = plan.M <= 64 ? TMG_PATH_SKINNY : TMG_PATH_TC;
    }

    switch (use) {
    case TMG_PATH_FFMA: {
        FfmaArgs a;
        a.A = A;
        a.B = B;
        a.D = D;
        a.la = to_dev(la);
        a.lb = to_dev(lb);
        a.ld = to_dev(ld);
        a.M = M;
        a.N = N;
        a.K = K;
        log_choice("%s %lldx%lldx%lld -> ffma_gemm_kernel (CUDA cores, operands read through their layouts)",
                   dt == 0 ? "f32" : "bf16", static_cast<long long>(M), static_cast<long long>(N),
                   static_cast<long long>(K));
        cudaError_t e = launch_ffma(a, dt, ds->num_sms, err_ctx(*ds), s);
        return e == cudaSuccess ? TMG_OK : cuda_fail(e, "ffma launch");
    }
    case TMG_PATH_TC:
    case TMG_PATH_TC_SINGLE:
    case TMG_PATH_TC_PAIR:
        if (dtype != TMG_BF16 || !plan.ok)
            return fail(TMG_ERR_UNSUPPORTED,
                        "tensor-core path needs bf16, K-major A and B (unit K stride, 16-byte aligned rows), "
                        "and row- or column-major D");
        return run_tc(*ds, plan, D, K, use == TMG_PATH_TC ? 0 : (use == TMG_PATH_TC_SINGLE ? 1 : 2), s);
    case TMG_PATH_SKINNY:
        if (dtype != TMG_BF16 || !plan.ok || plan.M > 64)
            return fail(TMG_ERR_UNSUPPORTED,
                        "skinny path needs bf16, K-major A and B, row- or column-major D, and at most 64 rows "
                        "on the small side");
        return run_skinny(*ds, plan, D, K, s);
    case TMG_PATH_PACKED_TC:
        if (dtype != TMG_BF16)
            return fail(TMG_ERR_UNSUPPORTED, "the general-layout tensor-core path takes bf16");
        log_choice("bf16 %lldx%lldx%lld -> general layouts on the tensor cores (operands the TMA cannot read in place "
                   "gathered through their layouts; the GEMM's own choice follows)",
                   static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K));
        return run_packed(*ds, A, B, D, M, N, K, la, lb, ld, s);
    case TMG_PATH_SKINNY_FFMA: {
        if (dtype != TMG_BF16 || !plan.ok || plan.M > 16 || K % 8 != 0)
            return fail(TMG_ERR_UNSUPPORTED,
                        "skinny FFMA path needs bf16, K-major A and B, K %% 8 == 0 and at most 16 rows");
        SkinnyFfmaArgs a{plan.A, plan.B, D, plan.M, plan.N, K, plan.lda, plan.ldb, plan.ldd};
        log_choice("bf16 %lldx%lldx%lld -> skinny_ffma_kernel (CUDA cores, warp-shuffle dot products)",
                   static_cast<long long>(plan.M), static_cast<long long>(plan.N), static_cast<long long>(K));
        cudaError_t e = launch_skinny_ffma(a, ds->num_sms, s);
        return e == cudaSuccess ? TMG_OK : cuda_fail(e, "skinny_ffma launch");
    }
    default:
        return fail(TMG_ERR_INVALID_ARG, "unknown path");
    }
}

tmg_status tmg_gemm(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, tmg_dtype dtype,
                    const tmg_layout *layoutA, const tmg_layout *layoutB, const tmg_layout *layoutD, void *stream)
{
    return tmg_gemm_ex(A, B, D, M, N, K, dtype, layoutA, layoutB, layoutD, TMG_PATH_AUTO, stream);
}

tmg_status tmg_gemm_host(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, tmg_dtype dtype,
                         void *stream)
{
    t_last_error.clear();
    if (dtype != TMG_F32 && dtype != TMG_BF16)
        return fail(TMG_ERR_INVALID_ARG, "tmg_gemm_host takes F32 or BF16 (got %d)", (int)dtype);
    if (M < 0 || N < 0 || K < 0)
        return fail(TMG_ERR_INVALID_ARG, "negative extent M=%lld N=%lld K=%lld", (long long)M, (long long)N,
                    (long long)K);
    if (M == 0 || N == 0)
        return TMG_OK;
    if (!D || (K > 0 && (!A || !B)))
        return fail(TMG_ERR_INVALID_ARG, "null operand pointer");
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    for (const void *p : {A, B, static_cast<const void *>(D)}) {
        cudaPointerAttributes pa;
        if (p && cudaPointerGetAttributes(&pa, p) == cudaSuccess && pa.type == cudaMemoryTypeDevice)
            return fail(TMG_ERR_INVALID_ARG, "tmg_gemm_host takes host buffers; %p is device memory", p);
        cudaGetLastError();
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t elem = dtype == TMG_F32 ? 4 : 2;
    const size_t bytes[3] = {static_cast<size_t>(M) * K * elem + 16, static_cast<size_t>(N) * K * elem + 16,
                             static_cast<size_t>(M) * N * elem};
    Scratch *sc = host_scratch(s, bytes, &st);
    if (!sc)
        return st;
    char *dA = static_cast<char *>(sc->host_ws[0]);
    char *dB = static_cast<char *>(sc->host_ws[1]);
    char *dD = static_cast<char *>(sc->host_ws[2]);
    cudaEvent_t *ev = sc->ev;
    // Row chunks of A and D: each chunk's copy in, GEMM and copy out run on
    // three streams, so chunk i's GEMM overlaps chunk i+1's upload and
    // chunk i-1's download.  Chunks are whole 256-row pair tiles.
    int64_t chunks = M / 512 > 0 ? M / 512 : 1;
    if (chunks > 16)
        chunks = 16;
    const int64_t rows_per = ((M + chunks - 1) / chunks + 255) / 256 * 256;
    chunks = (M + rows_per - 1) / rows_per;
    cudaError_t e;
    auto check = [&](cudaError_t r, const char *what) { return r == cudaSuccess ? TMG_OK : cuda_fail(r, what); };
    // the copies start after the work already queued on the caller's stream
    if ((st = check(cudaEventRecord(ev[0], s), "cudaEventRecord")) != TMG_OK ||
        (st = check(cudaStreamWaitEvent(sc->copy_in, ev[0], 0), "cudaStreamWaitEvent")) != TMG_OK ||
        (st = check(cudaStreamWaitEvent(sc->copy_out, ev[0], 0), "cudaStreamWaitEvent")) != TMG_OK)
        return st;
    if (K > 0 && (e = cudaMemcpyAsync(dB, B, static_cast<size_t>(N) * K * elem, cudaMemcpyHostToDevice,
                                      sc->copy_in)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync(B to device)");
    for (int64_t c = 0; c < chunks; ++c) {
        const int64_t m0 = c * rows_per, mc = (m0 + rows_per <= M ? rows_per : M - m0);
        cudaEvent_t in = ev[2 + 3 * c], done = ev[3 + 3 * c];
        if (K > 0 && (e = cudaMemcpyAsync(dA + m0 * K * elem, static_cast<const char *>(A) + m0 * K * elem,
                                          static_cast<size_t>(mc) * K * elem, cudaMemcpyHostToDevice,
                                          sc->copy_in)) != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyAsync(A rows to device)");
        if ((st = check(cudaEventRecord(in, sc->copy_in), "cudaEventRecord")) != TMG_OK ||
            (st = check(cudaStreamWaitEvent(s, in, 0), "cudaStreamWaitEvent")) != TMG_OK)
            return st;
        if ((st = tmg_gemm_ex(dA + m0 * K * elem, dB, dD + m0 * N * elem, mc, N, K, dtype, nullptr, nullptr,
                              nullptr, TMG_PATH_AUTO, s)) != TMG_OK)
            return st;
        if ((st = check(cudaEventRecord(done, s), "cudaEventRecord")) != TMG_OK ||
            (st = check(cudaStreamWaitEvent(sc->copy_out, done, 0), "cudaStreamWaitEvent")) != TMG_OK)
            return st;
        if ((e = cudaMemcpyAsync(static_cast<char *>(D) + m0 * N * elem, dD + m0 * N * elem,
                                 static_cast<size_t>(mc) * N * elem, cudaMemcpyDeviceToHost, sc->copy_out)) !=
            cudaSuccess)
            return cuda_fail(e, "cudaMemcpyAsync(D rows to host)");
    }
    // the caller's stream continues once D is back on the host
    if ((st = check(cudaEventRecord(ev[1], sc->copy_out), "cudaEventRecord")) != TMG_OK ||
        (st = check(cudaStreamWaitEvent(s, ev[1], 0), "cudaStreamWaitEvent")) != TMG_OK)
        return st;
    return TMG_OK;
}

tmg_status tmg_gemm_fused(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                          tmg_dtype in_dtype, const float *scale_a, const float *scale_b, const float *bias,
                          tmg_epilogue epilogue, void *stream)
{
    t_last_error.clear();
    if (in_dtype == TMG_F32)
        return fail(TMG_ERR_UNSUPPORTED, "the fused GEMM takes bf16 or E4M3 inputs (fp32 has no tensor-core path)");
    if (in_dtype != TMG_BF16 && in_dtype != TMG_E4M3)
        return fail(TMG_ERR_INVALID_ARG, "unknown input dtype %d", (int)in_dtype);
    if (epilogue < TMG_EPI_NONE || epilogue > TMG_EPI_BIAS_GELU)
        return fail(TMG_ERR_INVALID_ARG, "unknown epilogue %d", (int)epilogue);
    if (M < 0 || N < 0 || K < 0)
        return fail(TMG_ERR_INVALID_ARG, "negative extent M=%lld N=%lld K=%lld", (long long)M, (long long)N,
                    (long long)K);
    if (epilogue >= TMG_EPI_BIAS && !bias)
        return fail(TMG_ERR_INVALID_ARG, "epilogue %d adds a bias but bias is NULL", (int)epilogue);
    if (M == 0 || N == 0)
        return TMG_OK;
    if (!D || (K > 0 && (!A || !B)))
        return fail(TMG_ERR_INVALID_ARG, "null operand pointer");
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Tc2Epi epi{scale_a, scale_b, bias, static_cast<int>(epilogue), 0};
    if (K == 0) {
        cudaError_t e = launch_fused_k0(D, M, N, epi, s);
        return e == cudaSuccess ? TMG_OK : cuda_fail(e, "fused K=0 launch");
    }
    const bool e4m3 = in_dtype == TMG_E4M3;
    const int elem = e4m3 ? 1 : 2;
    if (!tma_ok(A, K, elem, M, K) || !tma_ok(B, K, elem, N, K) || M > INT32_MAX || N > INT32_MAX ||
        K > INT32_MAX)
        return fail(TMG_ERR_UNSUPPORTED, "the fused GEMM needs 16-byte aligned operands and rows (K * %d bytes "
                    "a multiple of 16)", elem);
    TcArgs a;
    std::memset(&a, 0, sizeof a);
    a.kb_elems = e4m3 ? 128 : 64;
    a.bn = pair_bn_override(tc2_pick_bn_of(M, N, K, a.kb_elems, ds->num_sms, kTc2FusedWidths, 4));
    const CUtensorMapDataType dt = e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if ((st = encode_2d(&a.tmA, dt, elem, A, K, M, K, a.kb_elems, 128)) != TMG_OK)
        return st;
    if ((st = encode_2d(&a.tmB, dt, elem, B, K, N, K, a.kb_elems, a.bn / 2)) != TMG_OK)
        return st;
    a.D = D;
    a.ldd = N;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    tc2_plan(a, ds->num_sms);
    int dev = 0;
    cudaGetDevice(&dev);
    if ((st = tc2_scratch(dev, s, a)) != TMG_OK)
        return st;
    log_choice("%s %dx%dx%d fused (epilogue %d, scale_a %s, scale_b %s) -> tc2_gemm_kernel (CTA pairs): 256x%d tiles, "
               "%d pairs, %d data-parallel + %d stream-K tiles, groups of %d M-tiles", e4m3 ? "e4m3" : "bf16", a.M, a.N,
               a.K, epi.epi, epi.scale_a ? "yes" : "no", epi.scale_b ? "yes" : "no", a.bn, a.pairs, a.dp_tiles,
               a.sk_tiles, a.group_m);
    cudaError_t e = launch_tc2_fused(a, epi, e4m3, err_ctx(*ds), s);
    return e == cudaSuccess ? TMG_OK : cuda_fail(e, "fused pair launch");
}

namespace {

// Both W4A8 entry points: B is the row-major packed int4 matrix, or (when
// `shuffled`) its pre-shuffled image.
tmg_status gemm_w4a8_impl(const void *A, const void *B, bool shuffled, void *D, int64_t M, int64_t N, int64_t K,
                          void *stream)
{
    t_last_error.clear();
    if (M < 0 || N < 0 || K < 0)
        return fail(TMG_ERR_INVALID_ARG, "negative extent M=%lld N=%lld K=%lld", (long long)M, (long long)N,
                    (long long)K);
    if (K % 2)
        return fail(TMG_ERR_INVALID_ARG, "K=%lld is odd (B packs two int4 values per byte)", (long long)K);
    if (shuffled && K % 32)
        return fail(TMG_ERR_INVALID_ARG, "K=%lld is not a multiple of 32 (pre-shuffled weights)", (long long)K);
    if (shuffled && reinterpret_cast<uintptr_t>(B) % 16)
        return fail(TMG_ERR_INVALID_ARG, "pre-shuffled weights not 16-byte aligned");
    if (M == 0 || N == 0)
        return TMG_OK;
    if (!D || (K > 0 && (!A || !B)))
        return fail(TMG_ERR_INVALID_ARG, "null operand pointer");
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return fail(TMG_ERR_UNSUPPORTED, "extents beyond 2^31");
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0) {
        e = cudaMemsetAsync(D, 0, static_cast<size_t>(M) * N * sizeof(int32_t), s);
        return e == cudaSuccess ? TMG_OK : cuda_fail(e, "cudaMemsetAsync(W4A8 D)");
    }
    // Decode shapes: the weights stay 4-bit until shared memory.
    bool decode = M <= 64 && K % 32 == 0 && K <= 32768;
    if (const char *f = getenv("TMG_W4A8_PATH")) {      // testing aid: "general" | "decode"
        if (!strcmp(f, "general"))
            decode = false;
    }
    if (decode && (shuffled || tma_ok(B, K / 2, 1, N, K / 2))) {
        W4a8SkinnyArgs w;
        std::memset(&w, 0, sizeof w);
        w.mp = static_cast<int>((M + 15) / 16 * 16);
        // A' (2 mp rows of K bytes), then the mp int32 row sums
        const size_t ap_bytes = static_cast<size_t>(2 * w.mp) * K;
        uint8_t *Ap = static_cast<uint8_t *>(pack_scratch(0, ap_bytes + 4 * static_cast<size_t>(w.mp), s, &st));
        if (!Ap)
            return st;
        if (shuffled)
            w.Bs = static_cast<const uint8_t *>(B);       // 1-D bulk copies; tmB stays unused
        else if ((st = encode_2d(&w.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K / 2, N, K / 2, 128, 128)) != TMG_OK)
            return st;
        if ((st = encode_2d(&w.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Ap, K, 2 * w.mp, K, 128, 2 * w.mp)) != TMG_OK)
            return st;
        w.grid = w4a8_skinny_grid(N, K, ds->num_sms);
        w.A = A;
        w.Ap = Ap;
        w.R = reinterpret_cast<int32_t *>(Ap + ap_bytes);
        w.D = static_cast<int32_t *>(D);
        w.ldd = N;
        w.M = static_cast<int>(M);
        w.N = static_cast<int>(N);
        w.K = static_cast<int>(K);
        log_choice("w4a8 %dx%dx%d -> split-activation pre-pass + w4a8_skinny_kernel (fp8 tensor cores, weights %s): "
                   "%d CTAs", w.M, w.N, w.K, w.Bs ? "pre-shuffled" : "row-major", w.grid);
        e = launch_w4a8_skinny(w, err_ctx(*ds), s);
        return e == cudaSuccess ? TMG_OK : cuda_fail(e, "W4A8 decode launch");
    }
    const int64_t ldp = (K + 7) / 8 * 8;
    void *PA = pack_scratch(0, static_cast<size_t>(M) * ldp * 2, s, &st);
    if (!PA)
        return st;
    void *PB = pack_scratch(1, static_cast<size_t>(N) * ldp * 2, s, &st);
    if (!PB)
        return st;
    if ((e = launch_unpack_w4a8(A, B, M, N, K, PA, PB, ldp, ds->num_sms, s, shuffled)) != cudaSuccess)
        return cuda_fail(e, "W4A8 unpack launch");
    // K segments of at most 8192: every partial sum of a segment is an integer
    // of magnitude <= 128 * 8 * 8192 = 2^23, exact in the fp32 accumulator
    // (integers up to 2^24 are); the first segment stores its int32 result,
    // the others add to it.
    constexpr int64_t kSeg = 8192;
    int dev = 0;
    cudaGetDevice(&dev);
    for (int64_t k0 = 0; k0 < K; k0 += kSeg) {
        const int64_t kc = K - k0 < kSeg ? K - k0 : kSeg;
        TcArgs a;
        std::memset(&a, 0, sizeof a);
        a.kb_elems = 64;
        a.bn = tc2_pick_bn_of(M, N, kc, 64, ds->num_sms, kTc2FusedWidths, 4);
        const uint16_t *pa = static_cast<const uint16_t *>(PA) + k0, *pb = static_cast<const uint16_t *>(PB) + k0;
        if ((st = encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pa, kc, M, ldp, 64, 128)) != TMG_OK)
            return st;
        if ((st = encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb, kc, N, ldp, 64, a.bn / 2)) != TMG_OK)
            return st;
        a.D = D;
        a.ldd = N;
        a.M = static_cast<int>(M);
        a.N = static_cast<int>(N);
        a.K = static_cast<int>(kc);
        tc2_plan(a, ds->num_sms);
        if ((st = tc2_scratch(dev, s, a)) != TMG_OK)
            return st;
        const Tc2Epi epi{nullptr, nullptr, nullptr, kEpiNone, k0 == 0 ? 1 : 2};
        log_choice("w4a8 %dx%dx%d, K segment at %lld -> tc2_gemm_kernel on the unpacked bf16 copies: 256x%d tiles, "
                   "%d pairs, groups of %d M-tiles, int32 %s", a.M, a.N, a.K, static_cast<long long>(k0), a.bn, a.pairs,
                   a.group_m, k0 == 0 ? "store" : "add");
        if ((e = launch_tc2_fused(a, epi, false, err_ctx(*ds), s)) != cudaSuccess)
            return cuda_fail(e, "W4A8 GEMM launch");
    }
    return TMG_OK;
}

}  // namespace

tmg_status tmg_gemm_w4a8(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *stream)
{
    return gemm_w4a8_impl(A, B, false, D, M, N, K, stream);
}

tmg_status tmg_gemm_w4a8_preshuffled(const void *A, const void *Bs, void *D, int64_t M, int64_t N, int64_t K,
                                     void *stream)
{
    return gemm_w4a8_impl(A, Bs, true, D, M, N, K, stream);
}

size_t tmg_w4a8_preshuffled_bytes(int64_t N, int64_t K)
{
    if (N <= 0 || K <= 0 || K % 32)
        return 0;
    return w4a8_preshuffled_bytes(N, K);
}

tmg_status tmg_w4a8_preshuffle(const void *B, void *Bs, int64_t N, int64_t K, void *stream)
{
    t_last_error.clear();
    if (N < 0 || K < 0)
        return fail(TMG_ERR_INVALID_ARG, "negative extent N=%lld K=%lld", (long long)N, (long long)K);
    if (K % 32)
        return fail(TMG_ERR_INVALID_ARG, "K=%lld is not a multiple of 32 (pre-shuffled weights)", (long long)K);
    if (N == 0 || K == 0)
        return TMG_OK;
    if (!B || !Bs)
        return fail(TMG_ERR_INVALID_ARG, "null pointer");
    if (reinterpret_cast<uintptr_t>(B) % 16 || reinterpret_cast<uintptr_t>(Bs) % 16)
        return fail(TMG_ERR_INVALID_ARG, "B and Bs must be 16-byte aligned");
    if (N > INT32_MAX || K > INT32_MAX)
        return fail(TMG_ERR_UNSUPPORTED, "extents beyond 2^31");
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    const cudaError_t e = launch_w4a8_preshuffle(B, N, K, Bs, ds->num_sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TMG_OK : cuda_fail(e, "W4A8 pre-shuffle launch");
}

tmg_status tmg_gemm_mxfp4(const void *A, const void *B, const void *scaleA, const void *scaleB, void *D, int64_t M,
                          int64_t N, int64_t K, void *stream)
{
    t_last_error.clear();
    if (M < 0 || N < 0 || K < 0)
        return fail(TMG_ERR_INVALID_ARG, "negative extent");
    if (K % 32 != 0)
        return fail(TMG_ERR_INVALID_ARG, "K=%lld is not a multiple of 32 (one e8m0 scale per 32 elements)",
                    (long long)K);
    if (M == 0 || N == 0)
        return TMG_OK;
    if (!D || (K > 0 && (!A || !B || !scaleA || !scaleB)))
        return fail(TMG_ERR_INVALID_ARG, "null operand pointer");
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        cudaError_t e = launch_zero_fill(D, to_dev(row_major(M, N)), M, N, 1, s);
        return e == cudaSuccess ? TMG_OK : cuda_fail(e, "zero_fill launch");
    }
    if (K % 256 != 0 || !tma_ok(A, K / 2, 1, M, K / 2) || !tma_ok(B, K / 2, 1, N, K / 2) || M > INT32_MAX ||
        N > INT32_MAX || K > INT32_MAX)
        return fail(TMG_ERR_UNSUPPORTED, "MXFP4 kernel needs K %% 256 == 0 and 16-byte aligned operand rows");
    if ((reinterpret_cast<uintptr_t>(scaleA) & 7u) || (reinterpret_cast<uintptr_t>(scaleB) & 7u))
        return fail(TMG_ERR_UNSUPPORTED, "MXFP4 scale arrays must be 8-byte aligned");
    Mxfp4Args a;
    std::memset(&a, 0, sizeof a);
    // CTA pairs once their tiles fill every SM pair; else one-CTA 128x128.
    bool pair = false;
    if (M >= 256) {
        a.bn = mxfp4_pair_pick_bn(M, N, ds->num_sms);
        pair = ((M + 255) / 256) * ((N + a.bn - 1) / a.bn) >= ds->num_sms / 2;
    }
    if (const char *f = getenv("TMG_MXFP4_KERNEL")) {        // testing aid: "single" | "pair"
        if (!strcmp(f, "single"))
            pair = false;
        else if (!strcmp(f, "pair") && M >= 256)
            pair = true;
        if (pair && a.bn == 0)
            a.bn = 128;
    }
    if (pair && getenv("TMG_MXFP4_BN"))
    {
        const int v = atoi(getenv("TMG_MXFP4_BN"));
        a.bn = (v == 128 || v == 256) ? v : 192;
    }
    const int box_b = pair ? a.bn / 2 : 128;
    if ((st = encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K / 2, M, K / 2, 128, 128)) != TMG_OK)
        return st;
    if ((st = encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K / 2, N, K / 2, 128, box_b)) != TMG_OK)
        return st;
    a.sA = static_cast<const uint8_t *>(scaleA);
    a.sB = static_cast<const uint8_t *>(scaleB);
    {
        int dev = 0;
        cudaGetDevice(&dev);
        const bool wide = pair && mxfp4_pair_wide_scales();
        const size_t ra = mxfp4_relaid_scale_bytes(M, K, 128, wide);
        const size_t rb = mxfp4_relaid_scale_bytes(N, K, pair ? a.bn : 128, wide);
        uint8_t *buf = mx_scale_scratch(dev, s, ra + rb, &st);
        if (!buf)
            return st;
        a.relA = buf;
        a.relB = buf + ra;
        if (pair) {
            const int nsub = (a.bn + 127) / 128;
            // one K block of one group's relaid scales, as rows of 256 bytes:
            // 4 KB (wide) or 1 KB (compact) per 128-row sub-block
            const int rows_per_sub = wide ? 16 : 4;
            if ((st = encode_2d(&a.tmSA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.relA, 256, ra / 256, 256, 256,
                                rows_per_sub, CU_TENSOR_MAP_SWIZZLE_NONE)) != TMG_OK)
                return st;
            if ((st = encode_2d(&a.tmSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.relB, 256, rb / 256, 256, 256,
                                rows_per_sub * nsub, CU_TENSOR_MAP_SWIZZLE_NONE)) != TMG_OK)
                return st;
        }
    }
    a.D = D;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    if (pair)
        log_choice("mxfp4 %dx%dx%d -> scale relayout + mxfp4_pair_kernel (CTA pairs): 256x%d tiles", a.M, a.N, a.K, a.bn);
    else
        log_choice("mxfp4 %dx%dx%d -> scale relayout + mxfp4_kernel (one CTA): 128x128 tiles", a.M, a.N, a.K);
    cudaError_t e = pair ? launch_mxfp4_pair(a, ds->num_sms, err_ctx(*ds), s) : launch_mxfp4(a, ds->num_sms, err_ctx(*ds), s);
    return e == cudaSuccess ? TMG_OK : cuda_fail(e, pair ? "mxfp4 pair launch" : "mxfp4 launch");
}

tmg_status tmg_gemm_skinny_noalloc(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                                   int64_t lda, int64_t ldb, int64_t ldd, void *stream)
{
    t_last_error.clear();
    if (M < 0 || N < 0 || K < 0)
        return fail(TMG_ERR_INVALID_ARG, "negative extent M=%lld N=%lld K=%lld", (long long)M, (long long)N,
                    (long long)K);
    if (M == 0 || N == 0)
        return TMG_OK;
    if (!D || (K > 0 && (!A || !B)))
        return fail(TMG_ERR_INVALID_ARG, "null operand pointer");
    if (M > 64)
        return fail(TMG_ERR_INVALID_ARG, "M=%lld exceeds the fixed-scratch skinny limit of 64 rows", (long long)M);
    if (ldd < N || (K > 0 && (lda < K || ldb < K)))
        return fail(TMG_ERR_INVALID_ARG, "leading dimension smaller than the row length");
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    FixedScratch fs;
    cudaError_t e = skinny_fixed_scratch(&fs);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(fixed skinny scratch)");
    const int64_t tiles = (N + 127) / 128;
    if (tiles > fs.max_tiles)
        return fail(TMG_ERR_INVALID_ARG, "N=%lld exceeds the fixed-scratch skinny limit of %lld", (long long)N,
                    (long long)fs.max_tiles * 128);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        tmg_layout ld = row_major(M, N);
        ld.stride[0][0] = ldd;
        e = launch_zero_fill(D, to_dev(ld), M, N, 1, s);
        return e == cudaSuccess ? TMG_OK : cuda_fail(e, "zero_fill launch");
    }
    if (!tma_ok(A, lda, 2, M, K) || !tma_ok(B, ldb, 2, N, K) || N > INT32_MAX || K > INT32_MAX)
        return fail(TMG_ERR_UNSUPPORTED, "operands need 16-byte aligned rows (row strides a multiple of 8)");
    SkinnyTcArgs a;
    std::memset(&a, 0, sizeof a);
    a.mp = static_cast<int>((M + 15) / 16 * 16);
    if ((st = encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, K, N, ldb, 64, 128)) != TMG_OK)
        return st;
    if ((st = encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, lda, 64, a.mp)) != TMG_OK)
        return st;
    const int64_t units = tiles * ((K + 63) / 64);
    const int64_t cap = static_cast<int64_t>(fs.partial_bytes / skinny_partials_bytes(1, a.mp));
    int64_t grid = ds->num_sms;
    if (units < grid)
        grid = units;
    if (cap < grid)
        grid = cap;
    a.grid = static_cast<int>(grid);
    a.partials = fs.partials;
    a.counters = fs.counters;
    a.D = D;
    a.ldd = ldd;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    // The array keeps the previous call's contents: the tile counters must
    // start at zero, the partial sums are always written before being read.
    if ((e = cudaMemsetAsync(fs.counters, 0, static_cast<size_t>(tiles) * 4 * sizeof(uint32_t), s)) != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(fixed skinny counters)");
    log_choice("bf16 %dx%dx%d -> skinny_tc_kernel with the fixed scratch array (MMA N = %d) on %d CTAs", a.M, a.N,
               a.K, a.mp, a.grid);
    e = launch_skinny_tc(a, err_ctx(*ds), s);
    return e == cudaSuccess ? TMG_OK : cuda_fail(e, "skinny_tc launch (fixed scratch)");
}

tmg_status tmg_check(void *stream)
{
    t_last_error.clear();
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    if ((e = cudaGetLastError()) != cudaSuccess)
        return cuda_fail(e, "pending CUDA error");
    uint32_t w = 0;
    if ((e = cudaMemcpy(&w, ds->err_word, sizeof w, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "reading the device error word");
    if (w != 0) {
        const bool bounds = (w & kErrBounds) != 0;
        cudaMemset(ds->err_word, 0, sizeof w);
        int dev = 0;
        cudaGetDevice(&dev);
        {
            std::lock_guard<std::mutex> lk(g_mu);
            for (auto &kv : g_scratch) {
                if (kv.first.first != dev)
                    continue;
                if (kv.second.counters)
                    cudaMemset(kv.second.counters, 0, kv.second.counters_bytes);
                if (kv.second.tc2_counters)
                    cudaMemset(kv.second.tc2_counters, 0, kv.second.tc2_counters_bytes);
            }
        }
        cudaDeviceSynchronize();
        if (bounds)
            return fail(TMG_ERR_BOUNDS, "a kernel computed an offset outside its buffer and skipped the access "
                                        "(error word 0x%08x, site %u)", w, w & 0xFFu);
        return fail(TMG_ERR_TIMEOUT, "a kernel wait ran out of its budget (error word 0x%08x, site %u)", w,
                    w & 0xFFu);
    }
    return TMG_OK;
}

const char *tmg_last_error(void) { return t_last_error.c_str(); }

void tmg_set_wait_budget_ns(uint64_t ns) { g_budget_ns.store(ns ? ns : 1); }

tmg_status tmg_debug_wait_timeout(uint64_t budget_ns, void *stream)
{
    t_last_error.clear();
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    ErrCtx ctx{ds->err_word, budget_ns};
    cudaError_t e = launch_wait_probe(ctx, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TMG_OK : cuda_fail(e, "wait probe launch");
}

tmg_status tmg_debug_bounds_probe(void *stream)
{
    t_last_error.clear();
#ifdef TMG_DEBUG_BOUNDS
    DeviceState *ds = nullptr;
    tmg_status st;
    if ((st = device_state(&ds)) != TMG_OK)
        return st;
    note_launch();
    bounds_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(1024, err_ctx(*ds));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TMG_OK : cuda_fail(e, "bounds probe launch");
#else
    (void)stream;
    return fail(TMG_ERR_UNSUPPORTED, "bounds checks exist only in the debug build (libtmg_debug.so)");
#endif
}

int tmg_debug_build(void)
{
#ifdef TMG_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

uint64_t tmg_launch_count(void) { return g_launches.load(); }

int tmg_version(void) { return 100; }

void tmg_shutdown(void)
{
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto &kv : g_scratch) {
        cudaSetDevice(kv.first.first);
        if (kv.second.partials)
            cudaFree(kv.second.partials);
        if (kv.second.counters)
            cudaFree(kv.second.counters);
        if (kv.second.mx_scales)
            cudaFree(kv.second.mx_scales);
        if (kv.second.tc2_partials)
            cudaFree(kv.second.tc2_partials);
        if (kv.second.tc2_counters)
            cudaFree(kv.second.tc2_counters);
        for (void *q : kv.second.pack)
            if (q)
                cudaFree(q);
        for (void *q : kv.second.host_ws)
            if (q)
                cudaFree(q);
        if (kv.second.copy_in) {
            cudaStreamSynchronize(kv.second.copy_in);
            cudaStreamSynchronize(kv.second.copy_out);
            cudaStreamDestroy(kv.second.copy_in);
            cudaStreamDestroy(kv.second.copy_out);
            for (cudaEvent_t ev : kv.second.ev)
                cudaEventDestroy(ev);
        }
    }
    g_scratch.clear();
    cudaSetDevice(cur);
    std::lock_guard<std::mutex> lk2(g_map_mu);
    g_maps.clear();
}

}  // extern "C"
