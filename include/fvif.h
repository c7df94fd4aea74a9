/*
 * fvif.h -- C ABI of libfvif, the 4-scale float VIF score on one GB300
 * (sm_103a) GPU.
 *
 * The score is the float_vif feature of a VMAF fork as its documentation
 * describes it:
 *   [A] "ADR-1422: float_vif_sycl computes the CPU's arithmetic without an
 *       fp64 type and returns its scores bit for bit", Context and Decision;
 *   [B] "ADR-1444: float_vif_hip runs the arithmetic of the CUDA twin from one
 *       shared header and returns the CPU's scores bit for bit", Context and
 *       Decision;
 *   [C] "Research-2130: float_ssim decimation on the SYCL device", Sources
 *       (picture_copy() sample normalisation).
 * For every frame pair it returns vif_scale0..3: four scales of separable
 * Gaussian filtering (taps computed at run time for (float)kernelscale) and
 * 2x decimation with a reflect-then-clamp boundary, per-pixel statistics,
 * two terms formed in fp64 and rounded once to fp32 before a polynomial
 * log2, and the per-scale ratio of two sequential fp32 sums (each row left
 * to right, then the row sums top to bottom).  Results are bit-identical to
 * the project's CPU oracle on every input.
 *
 * Conventions for every entry point:
 *  - Frames are luma planes, row-major, stride = w samples, n frames packed
 *    back to back.  Samples are uint8 when bitdepth == 8, else uint16 (host
 *    byte order); 9..16-bit samples are divided by 2^(bitdepth-8) ([C]).
 *    Sample values are not validated.
 *  - Scores are written frame-major: out[4*f + s] = vif_scale<s> of frame f.
 *  - Functions return FVIF_OK (0) or a negative status; on error the output
 *    contents are unspecified.  The status is also kept for
 *    fvif_last_error().
 *  - A context is not thread-safe; separate contexts are independent.
 *  - A pointer that is not a live context (destroyed, or never returned by
 *    fvif_create) is rejected with FVIF_EINVAL and never dereferenced;
 *    destroying it is a no-op.
 *  - All work runs on the context's CUDA stream (default: the legacy default
 *    stream; see fvif_set_stream).
 *
 * Environment variables read by the library (none is needed):
 *  - FVIF_LOG: when set, one line per create and score call on stderr (size,
 *    frames, chunk, status, host wall time; for fvif_score_async the time to
 *    enqueue).
 *  - FVIF_CHUNK=n: frames per chunk of device inputs (1..1024) instead of
 *    the default, read by fvif_create.
 *  - FVIF_TERMS=fp64: the two log terms of every pixel are evaluated by the
 *    fp64 sequence itself instead of fp32 pairs with an fp64 fallback (same
 *    bits, much slower; a check of the pair path), read by fvif_create.
 *  - FVIF_HOST_SLOTS=n (2..4, default 3) and FVIF_HOST_LANES=n (1..2,
 *    default 2): staging slots and compute lanes of fvif_score_host, read
 *    by fvif_create (tuning knobs; the defaults were measured best).
 *  - FVIF_DEC_TMA=0: the first decimation (integer samples to scale 1)
 *    loads its samples directly from global memory instead of staging each
 *    tile in shared memory by tensor copies (same bits; read once per
 *    process).  Staging is used when a frame's rows and the distance
 *    between frames are multiples of 16 bytes and the planes start on a
 *    16-byte boundary; a staged tile that has not arrived within one
 *    second makes its CTA give up and the next synchronous call on the
 *    context (fvif_score, fvif_score_host, fvif_score_debug) return
 *    FVIF_ECUDA.
 *  - FVIF_TEST_DEC_STALL=1: test hook, read by fvif_create: the staged
 *    decimation of that context waits for 16 bytes more than its tensor
 *    copies deliver, so every such wait runs into its one-second limit and
 *    the synchronous calls return FVIF_ECUDA (the timeout path, exercised
 *    without any fault).
 *  - FVIF_FAIL_ALLOC=n: test hook, read by fvif_create: allocation n
 *    (0 = the first) of the context fails as if the device were out of
 *    memory, so every failure path can be exercised without exhausting
 *    device memory.
 */
#ifndef FVIF_H
#define FVIF_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fvif_ctx fvif_ctx;

enum fvif_status {
    FVIF_OK = 0,
    FVIF_EINVAL = -1, /* invalid argument (size, bit depth, pointer, ...) */
    FVIF_ENOMEM = -2, /* device or pinned host allocation failed */
    FVIF_ECUDA = -3,  /* a CUDA call or kernel launch failed */
    FVIF_ETOOBIG = -4 /* frame too large for fvif_score_noalloc's scratch */
};

/* Create a context for frames of w x h samples.
 *  w, h        : 16 .. 16384 ([B] Context: frames down to 16x16 must run,
 *                including those under 72 px whose scale-3 planes are
 *                narrower than the filter).
 *  bitdepth    : 8 .. 16.
 *  kernelscale : > 0; used as a float ([A] Decision: taps for the float
 *                value of vif_kernelscale).  Scale s uses 2r+1 taps with
 *                r = floor(kernelscale * (2^(4-s)+1) / 2); r of scale 0 must
 *                not exceed 64.
 *  sigma_nsq   : > 0, finite; kept as a double ([A] Context: the noise
 *                variance stays fp64 in the statistic).
 * Allocates the pyramid and scratch buffers for one chunk of frames on the
 * current CUDA device.  Returns NULL on failure; the reason is then given by
 * fvif_last_error(NULL). */
fvif_ctx *fvif_create(int w, int h, int bitdepth, float kernelscale,
                      double sigma_nsq);

/* The extractor's options ("ADR-1422 ...", Decision and Consequences; "ADR-1444
 * ...", Consequences name vif_enhn_gain_limit, vif_skip_scale0 and
 * vif_scale1/2/3_min_val; their semantics here are this library's readings):
 *  enhn_gain_limit : cap on the gain g (default 100).
 *  skip_scale0     : nonzero -> scale 0 contributes nothing: its sums and
 *                    vif_scale0 are 0 (default 0).
 *  min_val[s]      : for s = 1..3, vif_scale_s = max(vif_scale_s, min_val[s])
 *                    (defaults 0; min_val[0] is ignored).
 *  frame_stride    : samples from the start of one input frame to the start
 *                    of the next (0 = w*h, planes packed back to back).  With
 *                    planar YUV frames (4:2:0, 4:2:2, 4:4:4) the luma plane
 *                    comes first, so the stride of the whole frame lets the
 *                    library read the luma planes in place: w*h*3/2, w*h*2
 *                    or w*h*3.  Must be 0 or >= w*h.  Applies to every
 *                    scoring entry point of the context; fvif_score_host
 *                    copies only the luma planes to the device. */
typedef struct fvif_options {
    float enhn_gain_limit;
    int skip_scale0;
    double min_val[4];
    long long frame_stride;
} fvif_options;

/* Fill *opt with the defaults above. */
void fvif_default_options(fvif_options *opt);

/* fvif_create with options (opt == NULL: defaults).  enhn_gain_limit must
 * be > 0 and finite, each min_val finite. */
fvif_ctx *fvif_create_ex(int w, int h, int bitdepth, float kernelscale,
                         double sigma_nsq, const fvif_options *opt);

/* Score n_frames frame pairs whose samples are in DEVICE memory (caller
 * owned, readable for the whole call; frames frame_stride samples apart,
 * see fvif_options).  out: HOST memory of 4*n_frames
 * doubles.  Synchronous: returns after out is written.  n_frames == 0 is a
 * no-op.  Frames are processed in chunks; no host round trip inside a
 * chunk. */
int fvif_score(fvif_ctx *ctx, const void *ref, const void *dist, int n_frames,
               double *out);

/* Same as fvif_score, but out is DEVICE memory of 4*n_frames doubles and the
 * call only enqueues work on the context stream (it returns before the
 * scores exist).  Inputs must stay valid until that stream reaches the end
 * of the enqueued work. */
int fvif_score_async(fvif_ctx *ctx, const void *ref, const void *dist,
                     int n_frames, double *out);

/* Score frame pairs whose samples are in HOST memory.  The library copies
 * chunks to the device on its own copy stream while earlier chunks are
 * scored (page-locked inputs overlap copy and compute; pageable ones still
 * work, slower).  out: HOST memory of 4*n_frames doubles.  Synchronous. */
int fvif_score_host(fvif_ctx *ctx, const void *ref, const void *dist,
                    int n_frames, double *out);

/* Page-locked HOST memory for the inputs of fvif_score_host: bytes rounded
 * up to 2 MiB, starting on a transparent-huge-page boundary (at least
 * 2 MiB), advised for huge pages and registered with the CUDA driver
 * (cudaHostRegister) on behalf of every device.  The copy engine moved
 * such buffers at the host link's full rate where large cudaHostAlloc
 * buffers varied by up to 9x.  The pages have no counterpart: this is a
 * host-memory helper of the library's input path.  Returns NULL if
 * bytes == 0 or on failure.  Free with fvif_host_free only. */
void *fvif_host_alloc(size_t bytes);

/* Release a buffer from fvif_host_alloc; NULL and unknown pointers are
 * ignored.  No call may still be using it. */
void fvif_host_free(void *p);

/* As fvif_score, with the fifteen debug outputs per frame in HOST memory
 * (out: 15*n_frames doubles, frame-major): vif_scale0..3, the frame ratio
 * vif = vif_num / vif_den, vif_num and vif_den (sums over the scales of the
 * per-scale sums, in fp64, scale 0 first), then num_scale0..3 and
 * den_scale0..3 (the per-scale fp32 sums).  "ADR-1444 ...", Consequences:
 * the debug mode emits fifteen outputs, the frame ratio and every per-scale
 * sum; the order and the fp64 totals are this library's reading. */
int fvif_score_debug(fvif_ctx *ctx, const void *ref, const void *dist,
                     int n_frames, double *out);

/* Free the context and everything it allocated.  NULL is a no-op. */
void fvif_destroy(fvif_ctx *ctx);

/* Run the context's work on cuda_stream (a cudaStream_t, or NULL for the
 * legacy default stream).  The stream stays owned by the caller. */
int fvif_set_stream(fvif_ctx *ctx, void *cuda_stream);

/* Status of the last call on ctx, or with ctx == NULL of the last
 * fvif_create on the calling thread. */
int fvif_last_error(const fvif_ctx *ctx);

/* Static text for a status code. */
const char *fvif_strerror(int status);

/* Number of frames the context scores per chunk of device inputs: enough
 * frames for about 4096 scale-0 strips of 16 rows per launch, at least 16
 * (31 at 3840x2160, 61 at 1920x1080).  fvif_score_host streams host inputs
 * in chunks of at most 16 frames. */
int fvif_chunk_frames(const fvif_ctx *ctx);

/* Copy the fp32 taps of scale s (0..3) into taps[0..cap); returns the tap
 * count, or a negative status. */
int fvif_get_taps(const fvif_ctx *ctx, int scale, float *taps, int cap);

/* Diagnostics for one frame pair (device inputs, host outputs), used to
 * localise a mismatch to one step.
 *  planes : the ref and dist planes of scales 0..3 as fp32, in the order
 *           ref0 dist0 ref1 dist1 ... (sum over s of 2 * w_s * h_s floats);
 *           may be NULL.
 *  rows   : per scale, the fp32 (num, den) sum of every row, scales one after
 *           another (sum over s of 2 * h_s floats); may be NULL.
 *  sums   : per scale the fp32 num and den totals (8 floats); may be NULL. */
int fvif_debug_frame(fvif_ctx *ctx, const void *ref, const void *dist,
                     float *planes, float *rows, float *sums);

/* The per-pixel statistic and terms of the context's kernels applied to n
 * given filtered statistics (mu1, mu2, xx, yy, xy; all DEVICE arrays of n
 * floats): num[i], den[i] receive the two log terms.  fallbacks (DEVICE,
 * may be NULL) is incremented once per pixel whose terms needed the native
 * fp64 sequence.  Enqueued on the context stream.  Diagnostics: checks the
 * term evaluation on arbitrary inputs. */
int fvif_debug_terms(fvif_ctx *ctx, const float *mu1, const float *mu2,
                     const float *xx, const float *yy, const float *xy,
                     int n, float *num, float *den,
                     unsigned long long *fallbacks);

/* Kernel kinds for the profiling counters. */
enum fvif_kernel_kind {
    FVIF_K_DECIMATE = 0, /* the three decimation launches of a chunk      */
    FVIF_K_STATS0 = 1,   /* the scale-0 statistic launch of a chunk       */
    FVIF_K_STATS123 = 2, /* the scale-1..3 statistic launches of a chunk  */
    FVIF_K_FINAL = 3,    /* the per-(frame, scale) final reduction        */
    FVIF_K_COUNT = 4
};

/* Opt-in per-kernel timing on the launching stream: while enabled, every
 * launch is bracketed by two CUDA events (the work itself is unchanged).
 * Enabling clears the counters. */
int fvif_profile_enable(fvif_ctx *ctx, int enable);

/* Total device time (ms, from the events) and launch count of one kernel
 * kind since profiling was enabled.  Waits for the recorded work to finish.
 * Launch counts are kept even when timing is disabled. */
int fvif_profile_read(fvif_ctx *ctx, int kind, double *total_ms,
                      long long *launches);

/* Per-chunk timing of the last fvif_score_host call made while profiling
 * was enabled (fvif_profile_enable), to show where a host-input call spends
 * its time: returns the number of chunks n of that call (0 if none) and
 * writes min(n, cap) rows of seven doubles to out (HOST memory):
 *   [0] copy start  : the chunk's host-to-device copy begins (its staging
 *                     slot is free and the copy stream reaches it),
 *   [1] copy end    : both of its planes are on the device,
 *   [2] score start : its lane may start it (copy done, lane free),
 *   [3] score end   : its scores are reduced,
 * all device time in ms since chunk 0's copy start (CUDA events), and
 *   [4], [5]        : host ms since the call began at which the library
 *                     started and finished enqueueing the chunk,
 *   [6]             : 1 if both of the chunk's input ranges were
 *                     page-locked for this process's CUDA runtime, else 0.
 * Waits for the recorded events.  Returns FVIF_EINVAL or FVIF_ECUDA on
 * error.  "ADR-1444 ...", Consequences, breaks the exact twin's frame time
 * down by measurement; this does the same for the host-input path. */
int fvif_profile_host(fvif_ctx *ctx, double *out, int cap);

/* Measured throughput of separately rounded fp32 multiplies and adds on
 * the current device, the operations the statistic is bound by ("ADR-1444
 * ...", Decision: every operation that rounds is written as one rounded
 * operation, so none is fused).  Runs one probe kernel on cuda_stream (NULL
 * = legacy default stream) in which every thread of 4 CTAs per SM steps 8
 * independent chains acc = acc * a + b (one rounded multiply, one rounded
 * add) iters times, as scalar operations (packed == 0) or as the packed
 * two-lane forms the filters use (packed != 0); waits for it and returns
 * the operation count in *ops and the event-timed duration in *ms.
 * Diagnostics for the roofline; allocates nothing.  FVIF_EINVAL for
 * iters <= 0 or NULL outputs, FVIF_ECUDA on a CUDA error. */
int fvif_alu_probe(int packed, long long iters, void *cuda_stream,
                   double *ops, double *ms);

/* Size in bytes of the fixed device scratch array used by
 * fvif_score_noalloc (8 MiB). */
#define FVIF_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/* Score frame pairs without allocating anything (no counterpart in the
 * pages: it exists for callers of this library that may not call cudaMalloc
 * -- code under a device memory arena or caching allocator that must own
 * every allocation, real-time loops that cannot take cudaMalloc's implicit
 * synchronisation, plug-ins with a fixed device-memory budget).
 *
 * Same arguments and results as fvif_create followed by fvif_score_async,
 * with no context: ref, dist (n_frames frames) and out (4*n_frames doubles)
 * are DEVICE memory owned by the caller; work is enqueued on cuda_stream
 * (NULL = legacy default stream) and the call returns without waiting.
 * Frames are scored one at a time through the same kernels as fvif_score,
 * with the intermediate planes and row sums kept in one file-scope device
 * array of FVIF_NOALLOC_SCRATCH_BYTES.  CUDA loads the library's device
 * code into a context lazily, so that array is taken from a device's memory
 * by the first call of this function there, and is held until the context
 * is destroyed or the process exits.  A caller with a fixed memory budget,
 * or one that captures streams into graphs, makes one call at set-up time,
 * before the budget is fixed and before any capture.
 *
 * Limit: a frame needs, rounding each part up to 256 bytes,
 * 8*(w1*h1) + 8*(w2*h2) + 8*(w3*h3) + 8*(h0+h1+h2+h3) bytes, where
 * w_s = w >> s and h_s = h >> s; frames whose need exceeds the array are
 * rejected with FVIF_ETOOBIG before anything is launched (1920x1080 needs
 * about 5.5 MB and fits; 3840x2160 does not).
 *
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress, a host-side lookup once the code is loaded), so
 * the call stays right after cudaDeviceReset or a change of context.  All
 * buffers must be on the current device.  Every call uses the same array and
 * leaves its
 * last contents there; nothing in it needs to start at zero.  Calls whose
 * work overlaps on the GPU (different streams, or several host threads)
 * race on the array: serialise them, e.g. on one stream.
 *
 * Returns FVIF_OK, FVIF_EINVAL (argument outside the ranges of
 * fvif_create, NULL buffer, negative count), FVIF_ETOOBIG or FVIF_ECUDA. */
int fvif_score_noalloc(int w, int h, int bitdepth, float kernelscale,
                       double sigma_nsq, const void *ref, const void *dist,
                       int n_frames, double *out, void *cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* FVIF_H */
