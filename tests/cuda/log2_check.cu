/* Test harness (not part of the library): the kernels' folded-range
 * division and packed log2 series, exhaustively on their domains. */
#include "../../vmaf_float_vif_gb300/csrc/fvif_kernels.cuh"

__global__ void div_check_kernel(unsigned lo, unsigned hi,
                                 unsigned long long *bad, unsigned *first)
{
    const unsigned bits = lo + blockIdx.x * blockDim.x + threadIdx.x;
    if (bits > hi)
        return;
    const float m = __uint_as_float(bits);
    const float a = __fsub_rn(m, 1.0f), b = __fadd_rn(m, 1.0f);
    const float q1 = fvif::div_folded(a, b);
    const float q2 = __fdiv_rn(a, b);
    if (__float_as_uint(q1) != __float_as_uint(q2)) {
        atomicAdd(bad, 1ull);
        atomicMin(first, bits);
    }
}

__global__ void log2_kernel(const float *x, int n, float *out, float2 one)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    /* lane 1 takes x[i], lane 2 takes x[n-1-i]: both lanes see every value */
    const float2 r = fvif::log2_series2(x[i], x[n - 1 - i], one);
    out[2 * (size_t)i] = r.x;
    out[2 * (size_t)(n - 1 - i) + 1] = r.y;
}

extern "C" int div_check(unsigned lo, unsigned hi, unsigned long long *bad_host,
                         unsigned *first_host)
{
    unsigned long long *bad;
    unsigned *first;
    if (cudaMalloc(&bad, sizeof *bad) != cudaSuccess)
        return -1;
    if (cudaMalloc(&first, sizeof *first) != cudaSuccess)
        return -1;
    cudaMemset(bad, 0, sizeof *bad);
    cudaMemset(first, 0xff, sizeof *first);
    const unsigned n = hi - lo + 1;
    div_check_kernel<<<(n + 255) / 256, 256>>>(lo, hi, bad, first);
    if (cudaGetLastError() != cudaSuccess)
        return -1;
    cudaMemcpy(bad_host, bad, sizeof *bad, cudaMemcpyDeviceToHost);
    cudaMemcpy(first_host, first, sizeof *first, cudaMemcpyDeviceToHost);
    cudaFree(bad);
    cudaFree(first);
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}

extern "C" int log2_eval(const float *x, int n, float *out)
{
    log2_kernel<<<(n + 255) / 256, 256>>>(x, n, out, make_float2(1.0f, 1.0f));
    if (cudaGetLastError() != cudaSuccess)
        return -1;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}
