/*
 * fssim_oracle.c -- plain CPU oracle for float_ssim's auto-scale decimation.
 *
 * TEST INFRASTRUCTURE ONLY, like the rest of this directory: nothing in the
 * product path links, loads or calls it, and it shares no code, header or
 * constant with the CUDA library.
 *
 * Source: "Research-2130: float_ssim decimation on the SYCL device"
 *  - Question: both planes are decimated by scale = max(1, round(min(w,h) /
 *    256)) before SSIM (4 at 1080p, 8 at 4K).
 *  - Sources: the low-pass kernel is scale x scale taps of 1.0f / (scale *
 *    scale) with the symmetric (period-2n mirror) boundary; output (x, y) of
 *    the decimation is the filtered value centred on sample (x * scale,
 *    y * scale), and the decimated size is w / scale + (w & 1) by
 *    h / scale + (h & 1); the filter's window offsets run from -k/2 to
 *    k/2 - 1 for even k and to k/2 for odd k; each fp32 product of sample and
 *    tap is added to a double sum, and the result is that sum times 1.0,
 *    rounded to float; 8-bit samples are taken as they are, 10/12/16-bit
 *    samples are divided by 4/16/256.
 *  - Findings, "The CPU sum is exact": for scale <= 128 every partial sum is
 *    exact in fp64, so the result is one round-to-nearest-even of the exact
 *    window sum; decimating in place gives the same planes as decimating
 *    from an untouched copy.
 *
 * Readings where the page leaves a step open:
 *  - round() is the C library's (half away from zero) of the real quotient
 *    min(w, h) / 256;
 *  - scale 1 leaves the plane as it is (the page's twins handled scale 1
 *    without a decimation; the size formula would otherwise add a column to
 *    odd widths);
 *  - the period-2n mirror maps j to j mod 2n, then to 2n - 1 - j when that is
 *    >= n (so -1 -> 0 and n -> n - 1, the edge sample repeated);
 *  - bit depths other than 8/10/12/16 divide by 2^(bitdepth - 8), as 10, 12
 *    and 16 do.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "fssim_oracle.h"

int fso_auto_scale(int w, int h)
{
    const int m = w < h ? w : h;
    const int s = (int)round((double)m / 256.0);
    return s > 1 ? s : 1;
}

int fso_mirror(int j, int n)
{
    const int p = 2 * n;
    int r = j % p;
    if (r < 0)
        r += p;
    return r >= n ? p - 1 - r : r;
}

int fso_out_size(int w, int h, int scale, int *sw, int *sh)
{
    if (w < 1 || h < 1 || scale < 1)
        return -1;
    if (scale == 1) {
        *sw = w;
        *sh = h;
    } else {
        *sw = w / scale + (w & 1);
        *sh = h / scale + (h & 1);
    }
    return 0;
}

float fso_tap(int scale)
{
    return 1.0f / (float)(scale * scale);
}

/* Sample normalisation: the value of sample i of a plane as fp32. */
static float sample_value(const void *plane, size_t i, int bitdepth)
{
    if (bitdepth == 8)
        return (float)((const uint8_t *)plane)[i];
    const float div = (float)(1 << (bitdepth - 8));
    return (float)((const uint16_t *)plane)[i] / div;
}

void fso_convert(const void *plane, int w, int h, int bitdepth, float *out)
{
    const size_t n = (size_t)w * (size_t)h;
    for (size_t i = 0; i < n; ++i)
        out[i] = sample_value(plane, i, bitdepth);
}

/* The filtered value centred on (cx, cy): the kernel's taps over the window,
 * fp32 products added to a double, rounded once to float at the end. */
static float filter_pixel(const float *img, int w, int h, int cx, int cy,
                          int k, float tap)
{
    const int lo = -(k / 2);
    const int hi = k / 2 - ((k % 2 == 0) ? 1 : 0);
    double sum = 0.0;
    for (int dy = lo; dy <= hi; ++dy) {
        const int yy = fso_mirror(cy + dy, h);
        for (int dx = lo; dx <= hi; ++dx) {
            const int xx = fso_mirror(cx + dx, w);
            const float prod = img[(size_t)yy * w + xx] * tap;
            sum += (double)prod;
        }
    }
    return (float)(sum * (double)1.0f);
}

int fso_decimate_plane(const float *img, int w, int h, int scale, float *out)
{
    int sw, sh;
    if (fso_out_size(w, h, scale, &sw, &sh) != 0)
        return -1;
    if (scale == 1) {
        for (size_t i = 0; i < (size_t)w * h; ++i)
            out[i] = img[i];
        return 0;
    }
    const float tap = fso_tap(scale);
    for (int y = 0; y < sh; ++y)
        for (int x = 0; x < sw; ++x)
            out[(size_t)y * sw + x] =
                filter_pixel(img, w, h, x * scale, y * scale, scale, tap);
    return 0;
}

int fso_decimate(const void *ref, const void *dist, int w, int h,
                 int bitdepth, int scale, int n_frames, float *ref_out,
                 float *dist_out, float *work)
{
    int sw, sh;
    if (bitdepth < 8 || bitdepth > 16 || scale < 1 ||
        fso_out_size(w, h, scale, &sw, &sh) != 0)
        return -1;
    const size_t in_elems = (size_t)w * h;
    const size_t in_bytes = in_elems * (bitdepth == 8 ? 1u : 2u);
    const size_t out_elems = (size_t)sw * sh;
    for (int f = 0; f < n_frames; ++f) {
        const unsigned char *r = (const unsigned char *)ref + in_bytes * f;
        const unsigned char *d = (const unsigned char *)dist + in_bytes * f;
        fso_convert(r, w, h, bitdepth, work);
        fso_decimate_plane(work, w, h, scale, ref_out + out_elems * f);
        fso_convert(d, w, h, bitdepth, work);
        fso_decimate_plane(work, w, h, scale, dist_out + out_elems * f);
    }
    return 0;
}
