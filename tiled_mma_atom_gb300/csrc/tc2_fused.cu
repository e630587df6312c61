// tc2_fused.cu — the pair kernel of tc2_kernel.cuh with the fused epilogue,
// for bf16 and E4M3 (kind::f8f6f4) inputs, and the K = 0 case of the fused
// GEMM.  Kept apart from tc2_bf16.cu so the two sets of instantiations
// compile in parallel.
#include "tc2_kernel.cuh"

namespace tmg {

const int kTc2FusedWidths[4] = {256, 224, 192, 128};

template <int IN>
static cudaError_t launch_fused_in(const TcArgs &a, const Tc2Epi &e, const ErrCtx &err, cudaStream_t s)
{
    switch (a.bn) {
    case 128:
        return launch_pair<128, IN, true>(a, e, err, s);
    case 192:
        return launch_pair<192, IN, true>(a, e, err, s);
    case 224:
        return launch_pair<224, IN, true>(a, e, err, s);
    case 256:
        return launch_pair<256, IN, true>(a, e, err, s);
    default:
        return cudaErrorInvalidValue;     // a width no kernel is built for
    }
}

cudaError_t launch_tc2_fused(const TcArgs &a, const Tc2Epi &e, bool in_e4m3, const ErrCtx &err, cudaStream_t s)
{
    return in_e4m3 ? launch_fused_in<kInE4m3>(a, e, err, s) : launch_fused_in<kInBf16>(a, e, err, s);
}

namespace {

__global__ void fused_k0_kernel(__nv_bfloat16 *__restrict__ D, int64_t M, int64_t N, Tc2Epi e)
{
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i % N;
        const float y = e.epi >= kEpiBias ? e.bias[n] : 0.f;
        // act(y) through the same arithmetic as the GEMM epilogue
        float r = y;
        if (e.epi == kEpiBiasRelu)
            r = fmaxf(y, 0.f);
        else if (e.epi == kEpiBiasSilu)
            r = __fdividef(y, 1.f + __expf(-y));
        else if (e.epi == kEpiBiasGelu)
            r = gelu_as(y);
        D[i] = __float2bfloat16_rn(r);
    }
}

}  // namespace

cudaError_t launch_fused_k0(void *D, int64_t M, int64_t N, const Tc2Epi &e, cudaStream_t s)
{
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096)
        blocks = 4096;
    note_launch();
    fused_k0_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<__nv_bfloat16 *>(D), M, N, e);
    return cudaGetLastError();
}

}  // namespace tmg
