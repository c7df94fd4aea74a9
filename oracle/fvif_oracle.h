/*
 * fvif_oracle.h -- declarations of the CPU oracle (test infrastructure only;
 * not part of the library and not shared with it).
 *
 * Samples: n frames, each w*h samples, row-major, stride w; uint8 when the
 * bit depth is 8, else uint16.  All buffers are host memory owned by the
 * caller.  Functions return 0 (or a tap count) on success, -1 on invalid
 * arguments, -2 on allocation failure.
 */
#ifndef FVIF_ORACLE_H
#define FVIF_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

#define FVO_MAX_TAPS 513
#define FVO_DEFAULT_GAIN_LIMIT 100.0f

int fvo_taps(float kernelscale, int scale, float *taps, int cap);
int fvo_mirror(int j, int n);
void fvo_filter(const float *src, int w, int h, const float *taps, int n,
                float *dst);
void fvo_decimate(const float *src, int w, int h, const float *taps, int n,
                  float *dst);
float fvo_log2f_approx(float x);
void fvo_pixel_terms(float mu1, float mu2, float xx, float yy, float xy,
                     double nsq, float gain_limit, float *num, float *den);
void fvo_log2f_approx_n(const float *x, int n, float *out);
void fvo_pixel_terms_n(const float *mu1, const float *mu2, const float *xx,
                       const float *yy, const float *xy, int n, double nsq,
                       float gain_limit, float *num, float *den);
int fvo_plane_size(int w, int h, int scale, int *ws, int *hs);
int fvo_frame_ex(const void *ref, const void *dist, int w, int h, int bd,
                 float kernelscale, double nsq, float gain_limit,
                 double *scores, float *rowsums, float *sums, float *planes);
int fvo_frame_opts(const void *ref, const void *dist, int w, int h, int bd,
                   float kernelscale, double nsq, float gain_limit,
                   int skip_scale0, const double *min_val, double *scores,
                   double *debug15);
int fvo_frame(const void *ref, const void *dist, int w, int h, int bd,
              float kernelscale, double nsq, double *scores);
int fvo_score(const void *ref, const void *dist, int w, int h, int bd,
              float kernelscale, double nsq, int n_frames, double *out);

#ifdef __cplusplus
}
#endif
#endif
