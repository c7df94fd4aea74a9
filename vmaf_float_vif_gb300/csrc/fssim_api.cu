/*
 * fssim_api.cu -- C ABI of float_ssim's auto-scale decimation (include/fssim.h):
 * argument checks, the tap's integer form and the launch shape.
 *
 * Source: "Research-2130: float_ssim decimation on the SYCL device" (Question:
 * scale = max(1, round(min(w, h) / 256)); Sources: tap 1.0f / (scale * scale),
 * decimated size w / scale + (w & 1) by h / scale + (h & 1); Findings, "The
 * CPU sum is exact": scales up to 128).
 */
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/fssim.h"
#include "fssim_kernels.cuh"

using namespace fssim;

namespace fssim {

FixedPath fixed_path_override()
{
    const char *v = std::getenv("FSSIM_KERNEL");
    if (!v)
        return FixedPath::kAuto;
    if (std::strcmp(v, "general") == 0)
        return FixedPath::kGeneral;
    if (std::strcmp(v, "windows") == 0)
        return FixedPath::kWindows;
    if (std::strcmp(v, "windows_direct") == 0)
        return FixedPath::kWindowsDirect;
    return FixedPath::kAuto;
}

/* FSSIM_TEST_STAGE_STALL=1 in the environment: the staged window kernel
 * waits for 16 bytes more than its copies bring, so its bounded wait runs
 * out and every block reads global memory instead (tests of that path). */
unsigned stage_extra_tx()
{
    const char *v = std::getenv("FSSIM_TEST_STAGE_STALL");
    return v && std::atoi(v) != 0 ? 16u : 0u;
}

} // namespace fssim

namespace {

bool valid_size(int w, int h)
{
    return w >= 1 && h >= 1 && w <= 16384 && h <= 16384;
}

} // namespace

extern "C" int fssim_auto_scale(int w, int h)
{
    if (!valid_size(w, h))
        return FVIF_EINVAL;
    const int m = w < h ? w : h;
    const int s = (int)std::round((double)m / 256.0);
    return s > 1 ? s : 1;
}

extern "C" int fssim_decimated_size(int w, int h, int scale, int *sw, int *sh)
{
    if (!valid_size(w, h) || scale < 0 || scale > FSSIM_MAX_SCALE || !sw ||
        !sh)
        return FVIF_EINVAL;
    if (scale == 0)
        scale = fssim_auto_scale(w, h);
    if (scale == 1) {
        *sw = w;
        *sh = h;
    } else {
        *sw = w / scale + (w & 1);
        *sh = h / scale + (h & 1);
    }
    return FVIF_OK;
}

extern "C" int fssim_decimate(int w, int h, int bitdepth, int scale,
                              const void *ref, const void *dist, int n_frames,
                              float *ref_out, float *dist_out,
                              void *cuda_stream)
{
    int sw = 0, sh = 0;
    if (bitdepth < 8 || bitdepth > 16 || n_frames < 0 ||
        fssim_decimated_size(w, h, scale, &sw, &sh) != FVIF_OK)
        return FVIF_EINVAL;
    if (n_frames > 0 && (!ref || !dist || !ref_out || !dist_out))
        return FVIF_EINVAL;
    const size_t B = bitdepth == 8 ? 1 : 2;
    if (n_frames > 0 &&
        (((uintptr_t)ref_out | (uintptr_t)dist_out) % 4 != 0 ||
         ((uintptr_t)ref | (uintptr_t)dist) % B != 0))
        return FVIF_EINVAL;
    if (n_frames == 0 || sw == 0 || sh == 0)
        return FVIF_OK;
    if (scale == 0)
        scale = fssim_auto_scale(w, h);
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    const int q = bitdepth - 8;
    const float inv_q = std::ldexp(1.0f, -q);

    if (scale == 1) {
        const size_t n = (size_t)w * h * (size_t)n_frames;
        const cudaError_t e =
            B == 1 ? convert<uint8_t>(ref, dist, ref_out, dist_out, n, inv_q,
                                      stream)
                   : convert<uint16_t>(ref, dist, ref_out, dist_out, n, inv_q,
                                       stream);
        return e == cudaSuccess ? FVIF_OK : FVIF_ECUDA;
    }

    const int k = scale;
    DecimateParams p = {};
    p.src[0] = ref;
    p.src[1] = dist;
    p.dst[0] = ref_out;
    p.dst[1] = dist_out;
    p.in_frame_elems = (size_t)w * h;
    p.out_frame_elems = (size_t)sw * sh;
    p.w = w;
    p.h = h;
    p.k = k;
    p.sw = sw;
    p.sh = sh;
    p.tap = 1.0f / (float)(k * k);
    int e2 = 0;
    const float mant = std::frexp(p.tap, &e2);       // tap = mant * 2^e2
    const int E = 24 - e2;                           // tap = T * 2^-E
    p.T = (long long)std::ldexp(mant, 24);
    p.err_scale = std::ldexp(1.0f, E);
    const bool exact = (k & (k - 1)) == 0;
    p.out_scale = exact ? p.tap * inv_q : std::ldexp(1.0f, -(q + E));
    p.packed16 = B == 2 && (long long)k * ((1 << bitdepth) - 1) < 65536;
    p.one2 = make_float2(1.0f, 1.0f);
    p.inv_q = inv_q;
    p.stage_extra_tx = stage_extra_tx();

    /* Tile: up to kMaxTileCols window columns (whole rows at 4K); shared
     * rows hold the groups of V columns those windows touch. */
    const int V = (int)(16 / B);
    p.X = sw < kMaxTileCols / k ? sw : kMaxTileCols / k;
    const long long span = (long long)p.X * k < w ? (long long)p.X * k : w;
    const int gmax = (int)((span + 2 * V - 2) / V);
    const int cols = gmax * V;
    p.pitch = cols + ((cols - 1) >> 5) + 1;
    /* Output rows per block: every thread of a group column walks at least
     * kBatch input rows (per threads share a column group when the tile has
     * fewer than kThreads groups); capped by shared memory. */
    const int per = kThreads / gmax > 0 ? kThreads / gmax : 1;
    int R = per * ((kBatch + k - 1) / k);
    const int words = exact ? 1 : 2;
    while (R > 1 && (size_t)R * p.pitch * sizeof(int) * words > kMaxSmem)
        --R;
    R = R > kMaxRows ? kMaxRows : R;
    p.R = R < sh ? R : sh;
    const size_t smem = (size_t)p.R * p.pitch * sizeof(int) * words;

    const bool vec = ((uintptr_t)ref % 16 == 0) &&
                     ((uintptr_t)dist % 16 == 0) && ((size_t)w * B) % 16 == 0;
    const cudaError_t e =
        B == 1 ? dispatch<uint8_t>(p, exact, vec, n_frames, smem, stream)
               : dispatch<uint16_t>(p, exact, vec, n_frames, smem, stream);
    return e == cudaSuccess ? FVIF_OK : FVIF_ECUDA;
}
