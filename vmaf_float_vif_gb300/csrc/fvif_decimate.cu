/* Decimation kernels, the per-(frame, scale) final reduction and the plane
 * unpacking used by the diagnostics entry point. */
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "fvif_dec_tma.cuh"
#include "fvif_dispatch.cuh"

namespace fvif {

namespace {

/* cuTensorMapEncodeTiled from the driver, looked up once through the
 * runtime (no link-time dependency on the driver library). */
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p,
                                             12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

/* FVIF_DEC_TMA=0 in the environment: the first decimation loads its
 * samples directly (decimate_kernel) instead of staging them by tensor
 * copies (same bits). */
bool dec_tma_enabled()
{
    static const bool on = [] {
        const char *e = std::getenv("FVIF_DEC_TMA");
        return !(e && std::atoi(e) == 0);
    }();
    return on;
}

/* A 3-D tensor map over n frames of one plane of integer samples: x (the
 * row, contiguous), y (rows, w apart), z (frames, frame_elems apart), with
 * the box of one decimation tile. */
bool make_plane_map(CUtensorMap *m, const void *base, SrcKind k, int w, int h,
                    int n, size_t frame_elems, int box_w, int box_h)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
    if (!enc)
        return false;
    const size_t eb = k == SrcKind::U8 ? 1 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)w, (cuuint64_t)h, (cuuint64_t)n};
    const cuuint64_t strides[2] = {(cuuint64_t)(w * eb),
                                   (cuuint64_t)(frame_elems * eb)};
    const cuuint32_t box[3] = {(cuuint32_t)box_w, (cuuint32_t)box_h, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m,
               k == SrcKind::U8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                : CU_TENSOR_MAP_DATA_TYPE_UINT16,
               3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

/* The staged variant serves a launch when: a status word is given, the
 * widths are fixed, the planes meet the tensor-copy rules (16-byte aligned
 * bases, rows and frames a multiple of 16 bytes apart) and are at least
 * 2R + 2 samples on each side (then every reflected index a kept output
 * needs lies inside its tile). */
template <int N, SrcKind K>
bool dec_tma_fits(const DecArgs &a)
{
    constexpr size_t eb = K == SrcKind::U8 ? 1 : 2;
    constexpr int r = N / 2;
    return a.status && dec_tma_enabled() && a.w >= 2 * r + 2 &&
           a.h >= 2 * r + 2 && (a.w * eb) % 16 == 0 &&
           (a.src.frame_elems * eb) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(a.src.x) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(a.src.y) % 16 == 0;
}

template <int N, SrcKind K>
cudaError_t run_decimate_tma(const DecArgs &a, const Taps &tp,
                             cudaStream_t st, bool *used)
{
    *used = false;
    constexpr int eb = K == SrcKind::U8 ? 1 : 2;
    constexpr int r = N / 2;
    if (!dec_tma_fits<N, K>(a))
        return cudaSuccess;
    CUtensorMap mx, my;
    if (!make_plane_map(&mx, a.src.x, K, a.w, a.h, a.nframes,
                        a.src.frame_elems, dtma_bw(r, eb), dtma_bh(r)) ||
        !make_plane_map(&my, a.src.y, K, a.w, a.h, a.nframes,
                        a.src.frame_elems, dtma_bw(r, eb), dtma_bh(r)))
        return cudaSuccess;
    static bool done[64];
    const int dx = dec_cols(r);
    const dim3 grid((unsigned)((a.w / 2 + dx - 1) / dx),
                    (unsigned)((a.h / 2 + kDY - 1) / kDY), (unsigned)a.nframes);
    const size_t bytes = dtma_smem_bytes(r, eb);
    cudaError_t e = ensure_smem(decimate_tma_kernel<N, K>, bytes, done);
    if (e != cudaSuccess)
        return e;
    decimate_tma_kernel<N, K><<<grid, kDecThreads, bytes, st>>>(mx, my, a, tp);
    *used = true;
    return cudaGetLastError();
}

} // namespace

cudaError_t stats_dispatch_u8(const StatsArgs &, const Taps &, cudaStream_t);
cudaError_t stats_dispatch_u16(const StatsArgs &, const Taps &, cudaStream_t);
cudaError_t stats_dispatch_f2(const StatsArgs &, const Taps &, cudaStream_t);

cudaError_t launch_stats(const StatsArgs &a, const Taps &tp, cudaStream_t st)
{
    switch (a.src.kind) {
    case SrcKind::U8: return stats_dispatch_u8(a, tp, st);
    case SrcKind::U16: return stats_dispatch_u16(a, tp, st);
    default: return stats_dispatch_f2(a, tp, st);
    }
}

template <int N, SrcKind K>
static cudaError_t dec_fixed_u(const DecArgs &a, const Taps &tp,
                               cudaStream_t st)
{
    bool used = false;
    const cudaError_t e = run_decimate_tma<N, K>(a, tp, st, &used);
    if (e != cudaSuccess || used)
        return e;
    return run_decimate<N, K>(a, tp, st);
}

template <SrcKind K>
static cudaError_t dec_dispatch_u(const DecArgs &a, const Taps &tp,
                                  cudaStream_t st)
{
    switch (tp.fixed_ok ? tp.n : 0) {
    case 5: return dec_fixed_u<5, K>(a, tp, st);
    case 9: return dec_fixed_u<9, K>(a, tp, st);
    case 19: return dec_fixed_u<19, K>(a, tp, st);
    default: return run_decimate<0, K>(a, tp, st);
    }
}

cudaError_t launch_decimate(const DecArgs &a, const Taps &tp, cudaStream_t st)
{
    switch (a.src.kind) {
    case SrcKind::U8: return dec_dispatch_u<SrcKind::U8>(a, tp, st);
    case SrcKind::U16: return dec_dispatch_u<SrcKind::U16>(a, tp, st);
    default:
        switch (tp.fixed_ok ? tp.n : 0) {
        case 1: return run_decimate<1, SrcKind::F2>(a, tp, st);
        case 3: return run_decimate<3, SrcKind::F2>(a, tp, st);
        case 5: return run_decimate<5, SrcKind::F2>(a, tp, st);
        case 7: return run_decimate<7, SrcKind::F2>(a, tp, st);
        case 11: return run_decimate<11, SrcKind::F2>(a, tp, st);
        default: return run_decimate<0, SrcKind::F2>(a, tp, st);
        }
    }
}

/* One warp per (frame, scale): the row sums added top to bottom into one
 * fp32 accumulator per output, then vif_scale = num / den in fp64
 * ("ADR-1422 ...", Decision: the rows' sums are added top to bottom in
 * fp32).  The warp stages 256 rows at a time in shared memory; lane 0 adds
 * them in order (the loads are independent of the sum chain, so they
 * pipeline). */
constexpr int kFinalWarps = 4;
constexpr int kFinalBatch = 256;

__global__ void __launch_bounds__(32 * kFinalWarps)
    final_kernel(const FinalArgs a)
{
    __shared__ float2 buf[kFinalWarps][kFinalBatch];
    const int wib = threadIdx.x >> 5;
    const int warp = blockIdx.x * kFinalWarps + wib;
    const int lane = threadIdx.x & 31;
    if (warp >= a.nframes * kScales)
        return;
    const int f = warp / kScales, s = warp % kScales;
    const bool skipped = (s == 0 && a.skip_scale0);
    const int h = skipped ? 0 : a.h[s];
    const float2 *r = a.rows + (size_t)f * a.rows_stride + a.rows_base[s];
    float num = 0.0f, den = 0.0f;
    for (int b = 0; b < h; b += kFinalBatch) {
        const int cnt = min(kFinalBatch, h - b);
        for (int j = lane; j < cnt; j += 32)
            buf[wib][j] = r[b + j];
        __syncwarp();
        if (lane == 0) {
#pragma unroll 8
            for (int j = 0; j < cnt; ++j) {
                const float2 v = buf[wib][j];
                num = __fadd_rn(num, v.x);
                den = __fadd_rn(den, v.y);
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        double score = skipped ? 0.0 : __ddiv_rn((double)num, (double)den);
        if (s > 0 && score < a.min_val[s])
            score = a.min_val[s];
        a.out[(size_t)f * kScales + s] = score;
        if (a.sums)
            a.sums[(size_t)f * kScales + s] = make_float2(num, den);
    }
}

/* One thread per frame: the fifteen debug values (see fvif_score_debug). */
__global__ void debug_kernel(const double *scores, const float2 *sums, int n,
                             double *out15)
{
    const int f = blockIdx.x * blockDim.x + threadIdx.x;
    if (f >= n)
        return;
    const float2 *sm = sums + (size_t)f * kScales;
    double *o = out15 + (size_t)f * 15;
    double num = 0.0, den = 0.0;
    for (int s = 0; s < kScales; ++s) {
        num = __dadd_rn(num, (double)sm[s].x);
        den = __dadd_rn(den, (double)sm[s].y);
    }
    for (int s = 0; s < kScales; ++s)
        o[s] = scores[(size_t)f * kScales + s];
    o[4] = __ddiv_rn(num, den);
    o[5] = num;
    o[6] = den;
    for (int s = 0; s < kScales; ++s) {
        o[7 + s] = (double)sm[s].x;
        o[11 + s] = (double)sm[s].y;
    }
}

cudaError_t launch_debug(const double *scores, const float2 *sums, int n,
                         double *out15, cudaStream_t st)
{
    debug_kernel<<<(n + 127) / 128, 128, 0, st>>>(scores, sums, n, out15);
    return cudaGetLastError();
}

cudaError_t launch_final(const FinalArgs &a, cudaStream_t st)
{
    const int warps = a.nframes * kScales;
    const int threads = 32 * kFinalWarps;
    const int blocks = (warps + kFinalWarps - 1) / kFinalWarps;
    final_kernel<<<blocks, threads, 0, st>>>(a);
    return cudaGetLastError();
}

__global__ void terms_kernel(const TermParams tp, const float *mu1,
                             const float *mu2, const float *xx,
                             const float *yy, const float *xy, int n,
                             float *num, float *den,
                             unsigned long long *fallbacks)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += gridDim.x * blockDim.x) {
        float a, b;
        if (fallbacks)
            pixel_terms<true>(mu1[i], mu2[i], xx[i], yy[i], xy[i], tp, a, b,
                              fallbacks);
        else
            pixel_terms<false>(mu1[i], mu2[i], xx[i], yy[i], xy[i], tp, a, b,
                               nullptr);
        num[i] = a;
        den[i] = b;
    }
}

cudaError_t launch_terms(const TermParams &tp, const float *mu1,
                         const float *mu2, const float *xx, const float *yy,
                         const float *xy, int n, float *num, float *den,
                         unsigned long long *fallbacks, cudaStream_t st)
{
    const int threads = 256;
    int blocks = (n + threads - 1) / threads;
    if (blocks > 152 * 32)
        blocks = 152 * 32;
    terms_kernel<<<blocks, threads, 0, st>>>(tp, mu1, mu2, xx, yy, xy, n, num,
                                             den, fallbacks);
    return cudaGetLastError();
}

template <SrcKind K>
__global__ void unpack_kernel(const SrcDesc d, int n, float *xo, float *yo)
{
    const Plane<K> p(d, 0);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += gridDim.x * blockDim.x) {
        const float2 v = p.at(i, d.scale);
        xo[i] = v.x;
        yo[i] = v.y;
    }
}

cudaError_t launch_unpack_planes(const SrcDesc &src, int w, int h,
                                 float *ref_out, float *dist_out,
                                 cudaStream_t st)
{
    const int n = w * h;
    const int blocks = (n + 255) / 256;
    switch (src.kind) {
    case SrcKind::U8:
        unpack_kernel<SrcKind::U8><<<blocks, 256, 0, st>>>(src, n, ref_out,
                                                           dist_out);
        break;
    case SrcKind::U16:
        unpack_kernel<SrcKind::U16><<<blocks, 256, 0, st>>>(src, n, ref_out,
                                                            dist_out);
        break;
    default:
        unpack_kernel<SrcKind::F2><<<blocks, 256, 0, st>>>(src, n, ref_out,
                                                           dist_out);
    }
    return cudaGetLastError();
}

} // namespace fvif
