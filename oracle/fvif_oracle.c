/*
 * fvif_oracle.c -- plain, slow CPU oracle for the 4-scale float VIF score.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * It is the definition the GPU library is checked against bit for bit: every
 * step is written as scalar loops in the order the method fixes, with every
 * fp32 operation rounded once (build with -ffp-contract=off, no fast-math).
 *
 * Sources (web pages of a VMAF fork's documentation):
 *  [A] "ADR-1422: float_vif_sycl computes the CPU's arithmetic without an
 *      fp64 type and returns its scores bit for bit" -- Context (table of the
 *      four properties: taps from vif_get_filter(), log2f_approx(),
 *      vif_sigma_nsq kept as a double, one fp32 sum per row then one over the
 *      rows; the two terms evaluated in fp64 and rounded once to fp32) and
 *      Decision (taps for (float)vif_kernelscale; the fp64 comparison of
 *      sigma1_sq with vif_sigma_nsq; row kernel adding left to right, rows
 *      added top to bottom).
 *  [B] "ADR-1444: float_vif_hip runs the arithmetic of the CUDA twin from one
 *      shared header and returns the CPU's scores bit for bit" -- Context
 *      (reflected tile index that must also be clamped; frames under 72 px)
 *      and Decision (decimate, per-pixel terms, per-row sums).
 *  [C] "Research-2130: float_ssim decimation on the SYCL device" -- Sources
 *      (picture_copy(): 8-bit samples as is, 10/12/16-bit divided by
 *      4/16/256).
 *  [D] "Research-1434: float_adm on SYCL without fp64" -- Findings, section 2
 *      (a default enhancement gain limit of 100).
 *
 * Readings where the pages leave a step open (each is one function below):
 *  - taps: the VIF Gaussian per scale (fvo_taps);
 *  - boundary: reflect about the edge sample once, then clamp (fvo_mirror);
 *  - filter: vertical pass first, then horizontal; each output is a
 *    sequential fp32 sum of fp32 products, tap 0 first (fvo_filter);
 *  - decimation: keep samples (2y, 2x), sizes halve with floor
 *    (fvo_decimate);
 *  - guards: the published VIF guards with eps = 1e-10f, and the
 *    low-variance rule for sigma1_sq < vif_sigma_nsq (fvo_pixel_terms);
 *  - log2f_approx: an atanh-series polynomial of our own (fvo_log2f_approx).
 *
 * Parity pins (tests, no GPU): tap symmetry and normalisation, the mirror
 * table, brute-force direct 2-D convolution, plane sizes, exact-rational
 * evaluation of the two fp64 term sequences, log2 error bounds, ref == dist
 * giving 1, flat frames giving exactly 1, and an fp64 textbook VIF within the
 * parity gate.  The low-variance constant and the guard order are pinned
 * only by those whole-score properties; agreement with upstream libvmaf's
 * numbers is unpinned (no golden scores are published).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "fvif_oracle.h"

#define NSCALES 4

/* ------------------------------------------------------------------------ */
/* Taps.  [A] Context + Decision: taps computed at run time for the float
 * value of vif_kernelscale.  Reading: scale s has the VIF base window
 * B = 2^(4-s) + 1 (17, 9, 5, 3) and Gaussian sigma = ks * B / 5; the
 * half-width is r = floor(ks * B / 2) in fp64, the width N = 2r + 1.
 * w_k = exp(-(k - r)^2 / (2 sigma^2)) in fp64, S = sum of w_k (k ascending,
 * fp64), tap_k = (float)(w_k / S).                                          */
int fvo_taps(float kernelscale, int scale, float *taps, int cap)
{
    if (scale < 0 || scale >= NSCALES || !(kernelscale > 0.0f))
        return -1;
    double base = (double)((1 << (4 - scale)) + 1);
    double ks = (double)kernelscale;
    double half = floor(ks * base / 2.0);
    if (half > 256.0)
        return -1;
    int r = (int)half;
    int n = 2 * r + 1;
    if (n > cap)
        return -1;
    if (r == 0) {
        taps[0] = 1.0f;
        return 1;
    }
    double sigma = ks * base / 5.0;
    double two_sigma_sq = 2.0 * sigma * sigma;
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    if (!w)
        return -1;
    double sum = 0.0;
    for (int k = 0; k < n; ++k) {
        double d = (double)(k - r);
        w[k] = exp(-(d * d) / two_sigma_sq);
        sum = sum + w[k];
    }
    for (int k = 0; k < n; ++k)
        taps[k] = (float)(w[k] / sum);
    free(w);
    return n;
}

/* ------------------------------------------------------------------------ */
/* Boundary.  [B] Context: an out-of-plane index is reflected and the result
 * must be clamped, so planes smaller than the filter stay in bounds.
 * Reading: mirror about the edge sample (no repeat), once, then clamp.      */
int fvo_mirror(int j, int n)
{
    if (j < 0)
        j = -j;
    else if (j >= n)
        j = 2 * (n - 1) - j;
    if (j < 0)
        j = 0;
    if (j > n - 1)
        j = n - 1;
    return j;
}

/* ------------------------------------------------------------------------ */
/* Separable filter, "same" size: vertical pass into tmp, then horizontal.   */
void fvo_filter(const float *src, int w, int h, const float *taps, int n,
                float *dst)
{
    int r = n / 2;
    float *tmp = (float *)malloc(sizeof(float) * (size_t)w * (size_t)h);
    if (!tmp)
        return;
    for (int i = 0; i < h; ++i) {
        for (int j = 0; j < w; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < n; ++k) {
                int ii = fvo_mirror(i + k - r, h);
                acc = acc + taps[k] * src[(size_t)ii * w + j];
            }
            tmp[(size_t)i * w + j] = acc;
        }
    }
    for (int i = 0; i < h; ++i) {
        for (int j = 0; j < w; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < n; ++k) {
                int jj = fvo_mirror(j + k - r, w);
                acc = acc + taps[k] * tmp[(size_t)i * w + jj];
            }
            dst[(size_t)i * w + j] = acc;
        }
    }
    free(tmp);
}

/* Decimation to the next scale: filter the whole plane with the next scale's
 * taps, then keep the samples at even row and even column ([B] Decision: a
 * decimate kernel per scale; sizes halve, rounding down).                   */
void fvo_decimate(const float *src, int w, int h, const float *taps, int n,
                  float *dst)
{
    int w2 = w / 2, h2 = h / 2;
    float *f = (float *)malloc(sizeof(float) * (size_t)w * (size_t)h);
    if (!f)
        return;
    fvo_filter(src, w, h, taps, n, f);
    for (int y = 0; y < h2; ++y)
        for (int x = 0; x < w2; ++x)
            dst[(size_t)y * w2 + x] = f[(size_t)(2 * y) * w + 2 * x];
    free(f);
}

/* ------------------------------------------------------------------------ */
/* log2f_approx.  [A] Context: the CPU takes log2 with a polynomial, not libm.
 * Ours (coefficients not on the pages): x = 2^e * m, m in [1, 2); if
 * m > fl32(sqrt 2) then m = m / 2, e = e + 1.  u = (m - 1) / (m + 1),
 * z = u * u, and log2 x ~ e + (2 / ln 2) * u * (1 + z/3 + z^2/5 + z^3/7 +
 * z^4/9)  (the atanh series), Horner in fp32, no fused operations.
 * Domain: finite normal x > 0 (the method only passes values >= 1).        */
float fvo_log2f_approx(float x)
{
    const float sqrt2 = 1.41421356237309515f;
    const float c9 = 1.0f / 9.0f;
    const float c7 = 1.0f / 7.0f;
    const float c5 = 1.0f / 5.0f;
    const float c3 = 1.0f / 3.0f;
    const float two_over_ln2 = (float)(2.0 / 0.69314718055994530942);
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    int e = (int)((bits >> 23) & 0xffu) - 127;
    uint32_t mbits = (bits & 0x007fffffu) | 0x3f800000u;
    float m;
    memcpy(&m, &mbits, sizeof m);
    if (m > sqrt2) {
        m = m * 0.5f;
        e = e + 1;
    }
    float u = (m - 1.0f) / (m + 1.0f);
    float z = u * u;
    float p = c9;
    p = c7 + z * p;
    p = c5 + z * p;
    p = c3 + z * p;
    p = 1.0f + z * p;
    float t = two_over_ln2 * u;
    t = t * p;
    return (float)e + t;
}

/* ------------------------------------------------------------------------ */
/* Per-pixel statistic and the two terms.
 * [A] Context: the two expressions 1 + (g*g*sigma1_sq)/(sv_sq + nsq) and
 * 1 + sigma1_sq/nsq are formed in fp64 (nsq is a double) and rounded to fp32
 * once, on the way into log2f_approx(); [A] Decision: the branch compares
 * sigma1_sq with nsq in fp64.  Guards, gain limit and the low-variance branch
 * are the published VIF ones (readings; [D] gives the default limit 100).  */
void fvo_pixel_terms(float mu1, float mu2, float xx, float yy, float xy,
                     double nsq, float gain_limit, float *num, float *den)
{
    const float eps = 1.0e-10f;
    const float lowvar_c = (float)(4.0 / (255.0 * 255.0));
    float s1 = xx - mu1 * mu1;
    float s2 = yy - mu2 * mu2;
    float s12 = xy - mu1 * mu2;
    s1 = s1 > 0.0f ? s1 : 0.0f;
    s2 = s2 > 0.0f ? s2 : 0.0f;
    float g = s12 / (s1 + eps);
    float sv = s2 - g * s12;
    if (s1 < eps) {
        g = 0.0f;
        sv = s2;
        s1 = 0.0f;
    }
    if (s2 < eps) {
        g = 0.0f;
        sv = 0.0f;
    }
    if (g < 0.0f) {
        sv = s2;
        g = 0.0f;
    }
    sv = sv > eps ? sv : eps;
    g = g < gain_limit ? g : gain_limit;

    if ((double)s1 < nsq) {
        *num = 1.0f - s2 * lowvar_c;
        *den = 1.0f;
    } else {
        float a = g * g * s1;
        double d = (double)sv + nsq;
        double q = (double)a / d;
        double v = 1.0 + q;
        *num = fvo_log2f_approx((float)v);
        double q2 = (double)s1 / nsq;
        double v2 = 1.0 + q2;
        *den = fvo_log2f_approx((float)v2);
    }
}

/* ------------------------------------------------------------------------ */
/* Ingest.  [C] Sources: 8-bit samples as they are; deeper samples are
 * uint16 divided by 2^(bitdepth - 8) (4, 16, 256 for 10, 12, 16 bits).      */
static void ingest(const void *src, int bd, size_t count, float *dst)
{
    if (bd == 8) {
        const uint8_t *p = (const uint8_t *)src;
        for (size_t i = 0; i < count; ++i)
            dst[i] = (float)p[i];
    } else {
        const uint16_t *p = (const uint16_t *)src;
        float scaler = (float)(1 << (bd - 8));
        for (size_t i = 0; i < count; ++i)
            dst[i] = (float)p[i] / scaler;
    }
}

int fvo_plane_size(int w, int h, int scale, int *ws, int *hs)
{
    if (scale < 0 || scale >= NSCALES)
        return -1;
    for (int s = 0; s < scale; ++s) {
        w = w / 2;
        h = h / 2;
    }
    *ws = w;
    *hs = h;
    return 0;
}

static int check_args(int w, int h, int bd, float ks, double nsq)
{
    if (w < 16 || h < 16 || w > 16384 || h > 16384)
        return -1;
    if (bd < 8 || bd > 16)
        return -1;
    if (!(ks > 0.0f) || !(nsq > 0.0))
        return -1;
    return 0;
}

/* One frame pair: four scales, per-scale rows, per-scale sums and score.
 * rowsums (optional): for each scale s, 2 * H_s floats (num, den per row),
 * scales one after another.  sums (optional): 8 floats, num_s and den_s.   */
int fvo_frame_ex(const void *ref, const void *dist, int w, int h, int bd,
                 float kernelscale, double nsq, float gain_limit,
                 double *scores, float *rowsums, float *sums, float *planes)
{
    if (check_args(w, h, bd, kernelscale, nsq))
        return -1;
    float taps[NSCALES][FVO_MAX_TAPS];
    int ntaps[NSCALES];
    for (int s = 0; s < NSCALES; ++s) {
        ntaps[s] = fvo_taps(kernelscale, s, taps[s], FVO_MAX_TAPS);
        if (ntaps[s] < 0)
            return -1;
    }
    size_t n0 = (size_t)w * (size_t)h;
    float *x = (float *)malloc(sizeof(float) * n0);
    float *y = (float *)malloc(sizeof(float) * n0);
    float *bufs = (float *)malloc(sizeof(float) * n0 * 8);
    float *nx = (float *)malloc(sizeof(float) * n0);
    float *ny = (float *)malloc(sizeof(float) * n0);
    if (!x || !y || !bufs || !nx || !ny) {
        free(x); free(y); free(bufs); free(nx); free(ny);
        return -2;
    }
    ingest(ref, bd, n0, x);
    ingest(dist, bd, n0, y);

    float *xx = bufs, *yy = bufs + n0, *xy = bufs + 2 * n0;
    float *mu1 = bufs + 3 * n0, *mu2 = bufs + 4 * n0;
    float *fxx = bufs + 5 * n0, *fyy = bufs + 6 * n0, *fxy = bufs + 7 * n0;

    int ws = w, hs = h;
    size_t rowoff = 0, planeoff = 0;
    for (int s = 0; s < NSCALES; ++s) {
        size_t np = (size_t)ws * (size_t)hs;
        if (planes) {
            memcpy(planes + planeoff, x, sizeof(float) * np);
            memcpy(planes + planeoff + np, y, sizeof(float) * np);
            planeoff += 2 * np;
        }
        for (size_t i = 0; i < np; ++i) {
            xx[i] = x[i] * x[i];
            yy[i] = y[i] * y[i];
            xy[i] = x[i] * y[i];
        }
        fvo_filter(x, ws, hs, taps[s], ntaps[s], mu1);
        fvo_filter(y, ws, hs, taps[s], ntaps[s], mu2);
        fvo_filter(xx, ws, hs, taps[s], ntaps[s], fxx);
        fvo_filter(yy, ws, hs, taps[s], ntaps[s], fyy);
        fvo_filter(xy, ws, hs, taps[s], ntaps[s], fxy);

        float total_num = 0.0f, total_den = 0.0f;
        for (int i = 0; i < hs; ++i) {
            float row_num = 0.0f, row_den = 0.0f;
            for (int j = 0; j < ws; ++j) {
                size_t p = (size_t)i * ws + j;
                float tn, td;
                fvo_pixel_terms(mu1[p], mu2[p], fxx[p], fyy[p], fxy[p], nsq,
                                gain_limit, &tn, &td);
                row_num = row_num + tn;
                row_den = row_den + td;
            }
            if (rowsums) {
                rowsums[rowoff + 2 * (size_t)i] = row_num;
                rowsums[rowoff + 2 * (size_t)i + 1] = row_den;
            }
            total_num = total_num + row_num;
            total_den = total_den + row_den;
        }
        rowoff += 2 * (size_t)hs;
        if (sums) {
            sums[2 * s] = total_num;
            sums[2 * s + 1] = total_den;
        }
        scores[s] = (double)total_num / (double)total_den;

        if (s + 1 < NSCALES) {
            int w2 = ws / 2, h2 = hs / 2;
            fvo_decimate(x, ws, hs, taps[s + 1], ntaps[s + 1], nx);
            fvo_decimate(y, ws, hs, taps[s + 1], ntaps[s + 1], ny);
            memcpy(x, nx, sizeof(float) * (size_t)w2 * (size_t)h2);
            memcpy(y, ny, sizeof(float) * (size_t)w2 * (size_t)h2);
            ws = w2;
            hs = h2;
        }
    }
    free(x); free(y); free(bufs); free(nx); free(ny);
    return 0;
}

/* The extractor's options and debug outputs.  "ADR-1422 ...", Decision and
 * Consequences, and "ADR-1444 ...", Consequences, name the option table
 * (vif_enhn_gain_limit, vif_skip_scale0, vif_scale1/2/3_min_val) and a
 * debug mode with fifteen outputs, the frame ratio and every per-scale sum;
 * their semantics are readings:
 *  - skip_scale0: scale 0 contributes nothing: num_0 = den_0 = 0 and
 *    vif_scale0 = 0 (scale 1 is still decimated from the scale-0 plane);
 *  - min_val[s] (s = 1..3): vif_scale_s = max(vif_scale_s, min_val[s]);
 *  - debug (15 doubles): vif_scale0..3 (floored), vif = vif_num / vif_den,
 *    vif_num = sum over s of num_s, vif_den likewise (fp64, s ascending),
 *    then num_0..3 and den_0..3 (the per-scale fp32 sums). */
int fvo_frame_opts(const void *ref, const void *dist, int w, int h, int bd,
                   float kernelscale, double nsq, float gain_limit,
                   int skip_scale0, const double *min_val, double *scores,
                   double *debug15)
{
    float sums[8];
    double raw[4];
    int rc = fvo_frame_ex(ref, dist, w, h, bd, kernelscale, nsq, gain_limit,
                          raw, NULL, sums, NULL);
    if (rc)
        return rc;
    if (skip_scale0) {
        sums[0] = 0.0f;
        sums[1] = 0.0f;
        raw[0] = 0.0;
    }
    for (int s = 0; s < NSCALES; ++s) {
        double v = raw[s];
        if (s > 0 && min_val && v < min_val[s])
            v = min_val[s];
        scores[s] = v;
    }
    if (debug15) {
        double num = 0.0, den = 0.0;
        for (int s = 0; s < NSCALES; ++s) {
            num = num + (double)sums[2 * s];
            den = den + (double)sums[2 * s + 1];
        }
        for (int s = 0; s < NSCALES; ++s)
            debug15[s] = scores[s];
        debug15[4] = num / den;
        debug15[5] = num;
        debug15[6] = den;
        for (int s = 0; s < NSCALES; ++s) {
            debug15[7 + s] = (double)sums[2 * s];
            debug15[11 + s] = (double)sums[2 * s + 1];
        }
    }
    return 0;
}

int fvo_frame(const void *ref, const void *dist, int w, int h, int bd,
              float kernelscale, double nsq, double *scores)
{
    return fvo_frame_ex(ref, dist, w, h, bd, kernelscale, nsq,
                        FVO_DEFAULT_GAIN_LIMIT, scores, NULL, NULL, NULL);
}

int fvo_score(const void *ref, const void *dist, int w, int h, int bd,
              float kernelscale, double nsq, int n_frames, double *out)
{
    if (n_frames < 0)
        return -1;
    size_t bytes = (size_t)w * (size_t)h * (bd == 8 ? 1u : 2u);
    for (int f = 0; f < n_frames; ++f) {
        int rc = fvo_frame((const char *)ref + bytes * (size_t)f,
                           (const char *)dist + bytes * (size_t)f, w, h, bd,
                           kernelscale, nsq, out + 4 * (size_t)f);
        if (rc)
            return rc;
    }
    return 0;
}

/* Array forms for tests: one call for many independent inputs. */
void fvo_log2f_approx_n(const float *x, int n, float *out)
{
    for (int i = 0; i < n; ++i)
        out[i] = fvo_log2f_approx(x[i]);
}

void fvo_pixel_terms_n(const float *mu1, const float *mu2, const float *xx,
                       const float *yy, const float *xy, int n, double nsq,
                       float gain_limit, float *num, float *den)
{
    for (int i = 0; i < n; ++i)
        fvo_pixel_terms(mu1[i], mu2[i], xx[i], yy[i], xy[i], nsq, gain_limit,
                        num + i, den + i);
}
