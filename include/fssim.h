/*
 * fssim.h -- C ABI of float_ssim's auto-scale decimation on the GPU (part of
 * libfvif.so; status codes are those of fvif.h).
 *
 * The operation is defined in "Research-2130: float_ssim decimation on the
 * SYCL device":
 *  - Question: float_ssim decimates both planes of a frame pair by
 *    scale = max(1, round(min(w, h) / 256)) before its SSIM stage (4 at
 *    1080p, 8 at 4K);
 *  - Sources: samples are converted as 8-bit values as they are and deeper
 *    samples divided by 2^(bitdepth - 8); the low-pass kernel is
 *    scale x scale taps of 1.0f / (scale * scale) with the symmetric
 *    (period-2n mirror) boundary; output (x, y) is the window centred on
 *    sample (x * scale, y * scale), offsets -scale/2 .. scale/2 - 1 for even
 *    scales and -scale/2 .. scale/2 for odd ones; each fp32 product of sample
 *    and tap enters a double sum that is rounded once to float; the
 *    decimated plane is w / scale + (w & 1) by h / scale + (h & 1);
 *  - Findings, "The CPU sum is exact": up to scale 128 that double sum is
 *    exact, so each output is the exact window sum rounded once to fp32.
 * This library reaches the same bits without fp64: the sample sums are
 * integers, and the rounding error of each product is recovered exactly and
 * summed exactly.  The window total is then formed exactly (in int64, or at
 * scales up to 8 as an exact fp32 pair) and rounded once to fp32.
 *
 * Scale 1 is no decimation: the outputs are the converted samples, w x h.
 * These are readings of the page: (a) scale 1 means no decimation; (b)
 * round() rounds the real quotient half away from zero; (c) bit depths 9, 11,
 * 13, 14 and 15 divide by 2^(bitdepth - 8), as 10, 12 and 16 do.
 *
 * Environment:
 *  - FSSIM_KERNEL=general|windows|windows_direct forces the kernel that
 *    scales 2..8 on 16-byte rows use (the default picks per scale and sample
 *    size, as measured); windows_direct is the window kernel without staging
 *    its rows in shared memory (scale 3 stages them by default).  Every
 *    choice gives the same bits.
 *  - FSSIM_TEST_STAGE_STALL=1: test hook, read by every fssim_decimate call:
 *    the staged kernel waits for more bytes than its copies bring, so its
 *    wait runs out after one second and each block reads its rows from
 *    global memory instead, with the same bits.  Never set it otherwise.
 */
#ifndef FSSIM_H
#define FSSIM_H

#include "fvif.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest scale accepted (the page's exactness bound). */
#define FSSIM_MAX_SCALE 128

/* The auto scale max(1, round(min(w, h) / 256)); FVIF_EINVAL (negative) if
 * w or h is outside [1, 16384]. */
int fssim_auto_scale(int w, int h);

/* Decimated plane size for a scale (0 = the auto scale) into *sw, *sh.
 * Returns FVIF_OK, or FVIF_EINVAL for w or h outside [1, 16384], scale
 * outside [0, FSSIM_MAX_SCALE] or NULL outputs.  Either side may be 0 (a
 * scale wider than an even side). */
int fssim_decimated_size(int w, int h, int scale, int *sw, int *sh);

/*
 * Decimate n_frames frame pairs.
 *   w, h       frame size, each in [1, 16384].
 *   bitdepth   8..16: uint8 samples for 8, uint16 (little-endian) otherwise.
 *              Sample values above 2^bitdepth - 1 are not checked.
 *   scale      1..FSSIM_MAX_SCALE, or 0 for the auto scale.
 *   ref, dist  DEVICE pointers owned by the caller: n_frames contiguous
 *              frames of w*h samples each (row stride w).  Any alignment of
 *              the sample type; 16-byte aligned buffers with a row length
 *              that is a multiple of 16 bytes take the vector path.
 *   ref_out, dist_out
 *              DEVICE pointers owned by the caller, 4-byte aligned:
 *              n_frames contiguous fp32 planes of sw*sh values each (row
 *              stride sw), frame-major, as fssim_decimated_size gives.
 *   cuda_stream  the cudaStream_t to run on (NULL: the legacy default
 *              stream).
 * Asynchronous: the work is enqueued on cuda_stream and the call returns
 * without waiting.  It allocates nothing and keeps no state, so calls from
 * several threads or on several streams are independent.  Returns FVIF_OK,
 * FVIF_EINVAL for bad arguments (nothing enqueued), or FVIF_ECUDA when a
 * launch fails (earlier launches of the same call may have run; the outputs
 * are then unspecified).
 */
int fssim_decimate(int w, int h, int bitdepth, int scale, const void *ref,
                   const void *dist, int n_frames, float *ref_out,
                   float *dist_out, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* FSSIM_H */
