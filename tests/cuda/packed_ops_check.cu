/* Test harness (not part of the library): the kernels' packed two-lane
 * multiply (mul2_rn) and accumulate (acc2_rn) against the scalar
 * round-to-nearest intrinsics, alone and chained the way the filters chain
 * them (mac5 with taps from memory). */
#include "../../vmaf_float_vif_gb300/csrc/fvif_kernels.cuh"

__constant__ float2 c_taps[8];

__global__ void packed_check_kernel(const float *a, const float *b,
                                    const float *c, int n, int form,
                                    float *out, float2 one)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    const float2 A = make_float2(a[i], b[i]);
    const float2 B = make_float2(b[i], c[i]);
    float *o = out + 4 * (size_t)i;
    if (form == 0) { /* single operations */
        const float2 m2 = fvif::mul2_rn(A, B);
        const float2 s2 = fvif::acc2_rn(A, B, one);
        o[0] = m2.x; o[1] = m2.y;
        o[2] = __fmul_rn(A.x, B.x); o[3] = __fmul_rn(A.y, B.y);
        o[4 * (size_t)n + 0] = s2.x; o[4 * (size_t)n + 1] = s2.y;
        o[4 * (size_t)n + 2] = __fadd_rn(A.x, B.x);
        o[4 * (size_t)n + 3] = __fadd_rn(A.y, B.y);
        return;
    }
    /* form 1: mac5 chain with register operands, form 2: taps from memory */
    fvif::Acc5 m5;
    fvif::mac5(m5, true, A, A, A.x, B, B, B.x, one);
    float ax = __fmul_rn(A.x, B.x), ay = __fmul_rn(A.y, B.y);
    for (int k = 1; k < 8; ++k) {
        const float2 q = make_float2(a[(i + k) % n], c[(i + 3 * k) % n]);
        const float2 t = form == 2 ? c_taps[k] : A;
        fvif::mac5(m5, false, t, t, t.x, q, q, q.x, one);
        ax = __fadd_rn(ax, __fmul_rn(t.x, q.x));
        ay = __fadd_rn(ay, __fmul_rn(t.y, q.y));
    }
    o[0] = m5.a.x; o[1] = m5.a.y; o[2] = ax; o[3] = ay;
}

extern "C" int packed_check(const float *a, const float *b, const float *c,
                            int n, int form, float *out)
{
    float2 taps[8];
    for (int k = 0; k < 8; ++k)
        taps[k] = make_float2(0.03125f * (k + 1) + 0.001f,
                              0.03125f * (k + 1) + 0.001f);
    if (cudaMemcpyToSymbol(c_taps, taps, sizeof taps) != cudaSuccess)
        return -2;
    packed_check_kernel<<<(n + 255) / 256, 256>>>(a, b, c, n, form, out,
                                                  make_float2(1.0f, 1.0f));
    if (cudaGetLastError() != cudaSuccess)
        return -1;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}
