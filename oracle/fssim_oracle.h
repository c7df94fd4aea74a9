/*
 * fssim_oracle.h -- plain CPU oracle for float_ssim's auto-scale decimation
 * (test infrastructure only; see fssim_oracle.c).
 */
#ifndef FSSIM_ORACLE_H
#define FSSIM_ORACLE_H

/* max(1, round(min(w, h) / 256)) */
int fso_auto_scale(int w, int h);
/* period-2n symmetric mirror of index j into [0, n) */
int fso_mirror(int j, int n);
/* decimated plane size; scale 1 keeps w x h.  0, or -1 on bad arguments */
int fso_out_size(int w, int h, int scale, int *sw, int *sh);
/* the low-pass tap 1.0f / (scale * scale) */
float fso_tap(int scale);
/* one plane of samples (uint8 for bitdepth 8, else uint16) to fp32 */
void fso_convert(const void *plane, int w, int h, int bitdepth, float *out);
/* one fp32 plane decimated by scale (out holds the decimated size) */
int fso_decimate_plane(const float *img, int w, int h, int scale, float *out);
/* n_frames contiguous frame pairs; work holds w*h floats */
int fso_decimate(const void *ref, const void *dist, int w, int h,
                 int bitdepth, int scale, int n_frames, float *ref_out,
                 float *dist_out, float *work);

#endif
