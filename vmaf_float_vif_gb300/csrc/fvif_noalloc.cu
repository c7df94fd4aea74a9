/*
 * fvif_noalloc.cu -- fvif_score_noalloc: the 4-scale score without any
 * allocation.
 *
 * Who needs it: callers that are not allowed to call cudaMalloc at the point
 * where they want a score.  Examples are code running under a device memory
 * arena or pool that owns all allocations (a framework's caching allocator,
 * an inference server with a fixed memory budget), real-time loops where
 * cudaMalloc's implicit device synchronisation and unbounded latency are not
 * acceptable, and plug-ins that must not grow the process's device
 * footprint at run time.  fvif_create allocates the pyramid, row-sum and
 * staging buffers; this entry point instead keeps every intermediate in one
 * fixed array compiled into the library and uses the caller's input and
 * output buffers as they are.
 *
 * The array belongs to this file's device module.  CUDA loads a module into
 * a context lazily by default, so the 8 MiB are taken from a device the first
 * time this entry point runs there (the address lookup below loads the
 * module), and are then held until the context is destroyed or the process
 * exits.  A caller with a fixed budget makes one call at set-up time.
 */

#include "../../include/fvif.h"
#include "fvif_internal.h"

using namespace fvif;

namespace {

/* Scratch for one frame pair: the float2 (ref, dist) planes of scales 1..3
 * and the per-row (num, den) sums of all four scales. */
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[FVIF_NOALLOC_SCRATCH_BYTES];

size_t align256(size_t n) { return (n + 255u) & ~(size_t)255u; }

/* Device address of the scratch array in the current context.  Host code
 * cannot use the array's name as a device pointer, so the address is looked
 * up with cudaGetSymbolAddress.  The lookup is repeated on every call: it is
 * a host-side table lookup once the module is loaded, and it stays right
 * after cudaDeviceReset or when the caller switches contexts, where an
 * address kept from an earlier context would no longer be mapped. */
int scratch_address(unsigned char **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess ||
        p == nullptr)
        return FVIF_ECUDA;
    *out = static_cast<unsigned char *>(p);
    return FVIF_OK;
}

} // namespace

extern "C" int fvif_score_noalloc(int w, int h, int bitdepth,
                                  float kernelscale, double sigma_nsq,
                                  const void *ref, const void *dist,
                                  int n_frames, double *out,
                                  void *cuda_stream)
{
    if (w < 16 || h < 16 || w > 16384 || h > 16384)
        return FVIF_EINVAL;
    if (bitdepth < 8 || bitdepth > 16)
        return FVIF_EINVAL;
    if (!(kernelscale > 0.0f) || !(kernelscale < 1e30f))
        return FVIF_EINVAL;
    if (!(sigma_nsq > 0.0) || !(sigma_nsq < 1e300))
        return FVIF_EINVAL;
    if (n_frames < 0 || (n_frames > 0 && (!ref || !dist || !out)))
        return FVIF_EINVAL;

    Taps taps[kScales];
    int ws[kScales], hs[kScales];
    for (int s = 0; s < kScales; ++s) {
        ws[s] = s == 0 ? w : ws[s - 1] / 2;
        hs[s] = s == 0 ? h : hs[s - 1] / 2;
        if (make_taps(kernelscale, s, taps[s]) != FVIF_OK)
            return FVIF_EINVAL;
        set_sample_taps(taps[s], bitdepth);
    }

    /* layout of the scratch for one frame */
    size_t off[kScales] = {0, 0, 0, 0};
    size_t need = 0;
    for (int s = 1; s < kScales; ++s) {
        off[s] = need;
        need += align256(sizeof(float2) * (size_t)ws[s] * hs[s]);
    }
    int rows_base[kScales];
    int rows_total = 0;
    for (int s = 0; s < kScales; ++s) {
        rows_base[s] = rows_total;
        rows_total += hs[s];
    }
    const size_t rows_off = need;
    need += align256(sizeof(float2) * (size_t)rows_total);
    if (need > (size_t)FVIF_NOALLOC_SCRATCH_BYTES)
        return FVIF_ETOOBIG;
    if (n_frames == 0)
        return FVIF_OK;

    unsigned char *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != FVIF_OK)
        return st;
    float2 *pyr[kScales] = {nullptr};
    for (int s = 1; s < kScales; ++s)
        pyr[s] = reinterpret_cast<float2 *>(scratch + off[s]);
    float2 *rows = reinterpret_cast<float2 *>(scratch + rows_off);
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

    TermParams terms;
    make_term_params(sigma_nsq, 100.0f, kTermsPair, terms);

    SrcDesc s0;
    s0.kind = bitdepth == 8 ? SrcKind::U8 : SrcKind::U16;
    s0.scale = bitdepth == 8 ? 1.0f : 1.0f / (float)(1 << (bitdepth - 8));
    s0.frame_elems = (size_t)w * h;
    const size_t frame_bytes = (size_t)w * h * (bitdepth == 8 ? 1u : 2u);

    /* One frame at a time through the same kernels as fvif_score.  Every
     * scratch byte a kernel reads was written earlier in the same frame
     * (decimation writes the whole plane it produces; the statistic writes
     * every row sum the final reduction reads), so nothing needs clearing
     * between calls. */
    cudaError_t e = cudaSuccess;
    for (int f = 0; f < n_frames && e == cudaSuccess; ++f) {
        s0.x = static_cast<const unsigned char *>(ref) + frame_bytes * f;
        s0.y = static_cast<const unsigned char *>(dist) + frame_bytes * f;
        for (int s = 1; s < kScales && e == cudaSuccess; ++s) {
            DecArgs d;
            if (s == 1) {
                d.src = s0;
            } else {
                d.src.kind = SrcKind::F2;
                d.src.x = pyr[s - 1];
                d.src.y = nullptr;
                d.src.scale = 1.0f;
                d.src.frame_elems = (size_t)ws[s - 1] * hs[s - 1];
            }
            d.w = ws[s - 1];
            d.h = hs[s - 1];
            d.nframes = 1;
            d.dst = pyr[s];
            d.dst_frame_elems = (size_t)ws[s] * hs[s];
            e = launch_decimate(d, taps[s], stream);
        }
        for (int s = 0; s < kScales && e == cudaSuccess; ++s) {
            StatsArgs a;
            if (s == 0) {
                a.src = s0;
            } else {
                a.src.kind = SrcKind::F2;
                a.src.x = pyr[s];
                a.src.y = nullptr;
                a.src.scale = 1.0f;
                a.src.frame_elems = (size_t)ws[s] * hs[s];
            }
            a.w = ws[s];
            a.h = hs[s];
            a.nframes = 1;
            a.terms = terms;
            a.rows = rows;
            a.rows_stride = rows_total;
            a.rows_base = rows_base[s];
            e = launch_stats(a, taps[s], stream);
        }
        if (e == cudaSuccess) {
            FinalArgs fa = {};
            fa.rows = rows;
            fa.rows_stride = rows_total;
            for (int s = 0; s < kScales; ++s) {
                fa.rows_base[s] = rows_base[s];
                fa.h[s] = hs[s];
            }
            fa.nframes = 1;
            fa.out = out + (size_t)kScales * f;
            fa.sums = nullptr;
            e = launch_final(fa, stream);
        }
    }
    return e == cudaSuccess ? FVIF_OK : FVIF_ECUDA;
}
