/*
 * fvif_probe.cu -- fvif_alu_probe: the measured throughput of the operations
 * the score is made of, on the current GPU.
 *
 * The statistic is bound by separately rounded fp32 multiplies and adds
 * (the method rounds every product and every sum, so nothing may be fused
 * and nothing maps onto tensor cores).  Its roofline is therefore the rate
 * at which the SMs retire such operations.  This probe measures that rate
 * instead of deriving it from the SM count and clock: every thread runs
 * kChains independent chains of acc = (acc * a) + b, each step one rounded
 * multiply and one rounded add, written either as scalar operations or as
 * the packed two-lane forms the filters use.
 */
#include "../../include/fvif.h"
#include "fvif_kernels.cuh"

namespace {

using namespace fvif;

constexpr int kProbeThreads = 256;
constexpr int kProbeBlocksPerSm = 4;
constexpr int kChains = 8;

/* where a probe would store its sum if it ever equalled the marker value
 * (it cannot for these inputs; the store keeps the chains from being
 * optimised away) */
__device__ float g_probe_sink;

__global__ void __launch_bounds__(kProbeThreads)
    alu_probe_scalar(long long iters, float a, float b)
{
    float acc[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c)
        acc[c] = (float)(threadIdx.x + c);
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c)
            acc[c] = __fadd_rn(__fmul_rn(acc[c], a), b);
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kChains; ++c)
        s = __fadd_rn(s, acc[c]);
    if (s == 12345.678f)
        g_probe_sink = s;
}

__global__ void __launch_bounds__(kProbeThreads)
    alu_probe_packed(long long iters, float2 a, float2 b, float2 one)
{
    float2 acc[kChains / 2];
#pragma unroll
    for (int c = 0; c < kChains / 2; ++c)
        acc[c] = make_float2((float)(threadIdx.x + c), (float)(c + 1));
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains / 2; ++c)
            acc[c] = acc2_rn(mul2_rn(acc[c], a), b, one);
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kChains / 2; ++c)
        s = __fadd_rn(s, __fadd_rn(acc[c].x, acc[c].y));
    if (s == 12345.678f)
        g_probe_sink = s;
}

} // namespace

extern "C" int fvif_alu_probe(int packed, long long iters, void *cuda_stream,
                              double *ops, double *ms)
{
    if (iters <= 0 || !ops || !ms)
        return FVIF_EINVAL;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess)
        return FVIF_ECUDA;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    const unsigned grid = (unsigned)(sms * kProbeBlocksPerSm);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess)
        e = cudaEventCreate(&e1);
    if (e == cudaSuccess)
        e = cudaEventRecord(e0, st);
    if (e == cudaSuccess) {
        if (packed)
            alu_probe_packed<<<grid, kProbeThreads, 0, st>>>(
                iters, make_float2(0.999999f, 0.999998f),
                make_float2(1e-7f, 2e-7f), make_float2(1.0f, 1.0f));
        else
            alu_probe_scalar<<<grid, kProbeThreads, 0, st>>>(
                iters, 0.999999f, 1e-7f);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess)
        e = cudaEventRecord(e1, st);
    if (e == cudaSuccess)
        e = cudaEventSynchronize(e1);
    float t = 0.0f;
    if (e == cudaSuccess)
        e = cudaEventElapsedTime(&t, e0, e1);
    if (e0)
        cudaEventDestroy(e0);
    if (e1)
        cudaEventDestroy(e1);
    if (e != cudaSuccess)
        return FVIF_ECUDA;
    /* two rounded operations per chain step, kChains lanes of chains per
     * thread either way (the packed kernel runs kChains/2 two-lane chains) */
    *ops = 2.0 * kChains * (double)iters * grid * kProbeThreads;
    *ms = t;
    return FVIF_OK;
}
