/*
 * fvif_internal.h -- declarations shared by the library's translation units
 * (host API and kernel instantiations).  Not part of the public ABI.
 */
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fvif {

constexpr int kScales = 4;
constexpr int kMaxRadius = 64;               /* largest half-width accepted  */
constexpr int kMaxTaps = 2 * kMaxRadius + 1; /* 129                          */

constexpr int kMaxFixedTaps = 35; /* widest kernel compiled with fixed N */

/* Taps of one scale, handed to a launch by value (kernel parameter space),
 * so compile-time-indexed reads become constant-bank operands.            */
struct Taps {
    float t[kMaxTaps];
    float2 t2[kMaxTaps]; /* (t[k], t[k]) for the packed two-lane operations */
    /* Vertical-pass taps for 16-bit integer samples s = x * 2^q (fixed
     * widths): t * x and t * (s * 2^-q) are the same real product, so
     * fl(t * x) = fl((t * 2^-q) * s); likewise fl(t * fl(x * x)) =
     * fl((t * 2^-2q) * fl(s * s)) and the same for x * y.  The passes
     * over 16-bit samples (the scale-0 statistic and the first decimation)
     * read them without rescaling.                                         */
    float2 ra2[kMaxFixedTaps]; /* (t 2^-q, t 2^-q)     for (x, y)           */
    float2 rb2[kMaxFixedTaps]; /* (t 2^-2q, t 2^-2q)   for (x*x, y*y)       */
    float rc[kMaxFixedTaps];   /* t 2^-2q              for x*y              */
    /* The fixed-width kernels may be used: n <= kMaxFixedTaps, the taps
     * are exactly symmetric (t[k] == t[n-1-k]: those kernels form each
     * product of a sample with a tap pair once) and every prescaled tap is
     * a normal fp32 value (the identity above needs it).                  */
    int fixed_ok;
    float2 one2;         /* (1, 1), read at run time (see acc2_rn)          */
    int n;
};

/* Fill ra2 / rb2 / rc / fixed_ok of taps for samples of this bit depth. */
void set_sample_taps(Taps &t, int bitdepth);

/* Where the samples of one plane come from. */
enum class SrcKind { U8, U16, F2 };

struct SrcDesc {
    SrcKind kind;
    const void *x;     /* U8/U16: ref samples; F2: interleaved (ref, dist)  */
    const void *y;     /* U8/U16: dist samples; F2: unused                  */
    float scale;       /* U16: 2^-(bitdepth-8); otherwise 1                 */
    size_t frame_elems;/* samples per frame of this plane                   */
};

/* How the two fp64 terms are evaluated. */
enum TermsMode {
    kTermsPair = 0, /* fp32 pairs, native fp64 only where undecided */
    kTermsFp64 = 1  /* native fp64 on every log-branch pixel        */
};

/* Constants of the per-pixel statistic, derived once on the host from the
 * fp64 noise variance (make_term_params). */
struct TermParams {
    double nsq;       /* vif_sigma_nsq                                      */
    float gain_limit;
    float nsq_up;     /* smallest fp32 >= nsq: (double)s < nsq <=> s < nsq_up */
    float n_hi, n_lo; /* nsq = n_hi + n_lo + e, |e| <= 2^-48 nsq            */
    float rcp_n;      /* fl32(1 / n_hi)                                     */
    float inv_pow2;   /* 1 / nsq when nsq is a power of two, else 0         */
    float2 one2;      /* (1, 1), read at run time by the packed sums        */
    int mode;         /* TermsMode                                          */
};

/* Per-scale statistic launch: all frames of a chunk, one CTA per strip. */
struct StatsArgs {
    SrcDesc src;
    int w, h;          /* plane size at this scale                          */
    int nframes;
    TermParams terms;
    float2 *rows;      /* row sums, (num, den)                              */
    int rows_stride;   /* float2 per frame in rows                          */
    int rows_base;     /* offset of this scale inside a frame's rows        */
};

/* Decimation launch: plane s (w x h) -> plane s+1 (w/2 x h/2), float2. */
struct DecArgs {
    SrcDesc src;
    int w, h;
    int nframes;
    float2 *dst;
    size_t dst_frame_elems;
    /* device word that a decimation whose staged tile did not arrive in
     * time marks (bit 0); nullptr: that variant is not used */
    unsigned *status = nullptr;
    /* test hook: bytes the staged decimation's mbarrier expects beyond what
     * its tensor copies deliver (0; nonzero makes every wait time out) */
    unsigned extra_tx = 0;
};

/* Final per-(frame, scale) reduction over the row sums. */
struct FinalArgs {
    const float2 *rows;
    int rows_stride;
    int rows_base[kScales];
    int h[kScales];
    int nframes;
    double *out;       /* device, 4 per frame                               */
    float2 *sums;      /* optional device (num, den) per (frame, scale)     */
    int skip_scale0;   /* scale 0 not computed: its sums and score are 0    */
    double min_val[kScales]; /* floors on scales 1..3                       */
};

/* Taps of scale s for a kernelscale (host); FVIF_OK or FVIF_EINVAL. */
int make_taps(float kernelscale, int s, Taps &out);

/* Statistic constants for a noise variance (host).  mode is a TermsMode;
 * outside [2^-60, 2^60] the pair evaluation is not used. */
void make_term_params(double nsq, float gain_limit, int mode, TermParams &out);

/* Per-pixel terms over arrays (diagnostics); fallbacks may be null. */
cudaError_t launch_terms(const TermParams &tp, const float *mu1,
                         const float *mu2, const float *xx, const float *yy,
                         const float *xy, int n, float *num, float *den,
                         unsigned long long *fallbacks, cudaStream_t st);

cudaError_t launch_stats(const StatsArgs &a, const Taps &taps,
                         cudaStream_t st);
cudaError_t launch_decimate(const DecArgs &a, const Taps &taps,
                            cudaStream_t st);
cudaError_t launch_final(const FinalArgs &a, cudaStream_t st);
/* The fifteen debug outputs of n frames from their scores and sums. */
cudaError_t launch_debug(const double *scores, const float2 *sums, int n,
                         double *out15, cudaStream_t st);
cudaError_t launch_unpack_planes(const SrcDesc &src, int w, int h,
                                 float *ref_out, float *dist_out,
                                 cudaStream_t st);

} // namespace fvif
