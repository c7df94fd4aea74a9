/*
 * fssim_u8.cu -- the float_ssim decimation kernels for uint8_t samples (one
 * translation unit per sample type, so the two compile in parallel).
 */
#include "fssim_kernels.cuh"

namespace fssim {

template <>
cudaError_t dispatch<uint8_t>(const DecimateParams &p, bool exact, bool vec,
                          int n_frames, size_t smem, cudaStream_t stream)
{
    return dispatch_impl<uint8_t>(p, exact, vec, n_frames, smem, stream);
}

template <>
cudaError_t convert<uint8_t>(const void *ref, const void *dist, float *ref_out,
                         float *dist_out, size_t n, float inv,
                         cudaStream_t stream)
{
    const size_t blocks = (n + kThreads - 1) / kThreads;
    const unsigned grid = blocks < 152u * 32u ? (unsigned)blocks : 152u * 32u;
    ssim_convert_kernel<uint8_t><<<grid, kThreads, 0, stream>>>(
        static_cast<const uint8_t *>(ref), static_cast<const uint8_t *>(dist),
        ref_out, dist_out, n, inv);
    return cudaGetLastError();
}

} // namespace fssim
