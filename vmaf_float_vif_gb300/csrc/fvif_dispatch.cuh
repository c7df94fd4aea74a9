/*
 * fvif_dispatch.cuh -- launch helpers shared by the kernel translation units.
 */
#pragma once

#include "fvif_kernels.cuh"

namespace fvif {

/* Shared-memory opt-in for one kernel instantiation, once per device. */
template <typename Kern>
inline cudaError_t ensure_smem(Kern *k, size_t bytes, bool *done_per_device)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    if (done_per_device[dev])
        return cudaSuccess;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bytes);
    if (e == cudaSuccess)
        done_per_device[dev] = true;
    return e;
}

template <int N, SrcKind K>
cudaError_t run_stats(const StatsArgs &a, const Taps &tp, cudaStream_t st)
{
    static bool done[64];
    const int r = (N > 0) ? N / 2 : tp.n / 2;
    /* the attribute is set for the largest width this variant serves */
    const size_t max_bytes = stats_smem_bytes(N > 0 ? N / 2 : kMaxRadius);
    cudaError_t e = ensure_smem(stats_kernel<N, K>, max_bytes, done);
    if (e != cudaSuccess)
        return e;
    const int nstrips = (a.h + kTH - 1) / kTH;
    const unsigned grid = (unsigned)(nstrips * a.nframes);
    stats_kernel<N, K><<<grid, kThreads, stats_smem_bytes(r), st>>>(a, tp);
    return cudaGetLastError();
}

template <int N, SrcKind K>
cudaError_t run_decimate(const DecArgs &a, const Taps &tp, cudaStream_t st)
{
    static bool done[64];
    const int r = (N > 0) ? N / 2 : tp.n / 2;
    const size_t max_bytes = dec_smem_bytes(N > 0 ? N / 2 : kMaxRadius);
    cudaError_t e = ensure_smem(decimate_kernel<N, K>, max_bytes, done);
    if (e != cudaSuccess)
        return e;
    const int dx = dec_cols(r);
    const dim3 grid((unsigned)((a.w / 2 + dx - 1) / dx),
                    (unsigned)((a.h / 2 + kDY - 1) / kDY), (unsigned)a.nframes);
    decimate_kernel<N, K><<<grid, kDecThreads, dec_smem_bytes(r), st>>>(a, tp);
    return cudaGetLastError();
}

} // namespace fvif
