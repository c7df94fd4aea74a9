/*
 * fvif_api.cu -- host side of libfvif: context, taps, chunked launches and
 * the C ABI declared in include/fvif.h.
 */
#include <cfloat>
#include <cmath>
#include <chrono>
#include <cstdio>
#include <vector>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>

#include "../../include/fvif.h"
#include "fvif_internal.h"

using namespace fvif;

namespace {

constexpr int kDefaultChunk = 16;   /* smallest chunk, in frames       */
constexpr int kMaxChunk = 1024;     /* largest chunk, in frames        */
constexpr int kChunkCtas = 4096;    /* scale-0 CTAs per chunk wanted   */
constexpr int kLanes = 2; /* chunks alternate between two streams */
constexpr int kMaxStage = 4; /* host-input staging slots, at most */

thread_local int g_create_status = FVIF_OK;

/* Contexts made by fvif_create and not yet destroyed: every entry point
 * rejects any other pointer (a destroyed context, a stray value) with
 * FVIF_EINVAL instead of dereferencing it. */
std::mutex g_live_mutex;
std::unordered_set<const fvif_ctx *> g_live;

bool live(const fvif_ctx *c)
{
    if (!c)
        return false;
    std::lock_guard<std::mutex> lock(g_live_mutex);
    return g_live.count(c) != 0;
}

} // namespace

namespace fvif {

/* Taps of scale s for kernelscale ks.  "ADR-1422: float_vif_sycl computes
 * the CPU's arithmetic without an fp64 type ...", Decision: the taps are the
 * CPU routine's, computed at run time for (float)vif_kernelscale and handed
 * to every launch by value.  The routine is the VIF Gaussian: base window
 * B = 2^(4-s)+1, sigma = ks B / 5, half-width r = floor(ks B / 2), weights
 * exp(-d^2 / (2 sigma^2)) in fp64 normalised by their fp64 sum (ascending),
 * each rounded to fp32.                                                     */
int make_taps(float kernelscale, int s, Taps &out)
{
    const double ks = (double)kernelscale;
    const double base = (double)((1 << (4 - s)) + 1);
    const double half = std::floor(ks * base / 2.0);
    if (!(half >= 0.0) || half > (double)kMaxRadius)
        return FVIF_EINVAL;
    const int r = (int)half;
    std::memset(&out, 0, sizeof out);
    out.n = 2 * r + 1;
    out.one2 = make_float2(1.0f, 1.0f);
    if (r == 0) {
        out.t[0] = 1.0f;
        out.t2[0] = make_float2(1.0f, 1.0f);
        return FVIF_OK;
    }
    const double sigma = ks * base / 5.0;
    const double two_sigma_sq = 2.0 * sigma * sigma;
    double wk[kMaxTaps];
    double sum = 0.0;
    for (int k = 0; k < out.n; ++k) {
        const double d = (double)(k - r);
        wk[k] = std::exp(-(d * d) / two_sigma_sq);
        sum = sum + wk[k];
    }
    for (int k = 0; k < out.n; ++k)
        out.t[k] = (float)(wk[k] / sum);
    for (int k = 0; k < out.n; ++k)
        out.t2[k] = make_float2(out.t[k], out.t[k]);
    set_sample_taps(out, 8);
    return FVIF_OK;
}

void set_sample_taps(Taps &t, int bitdepth)
{
    const int q = bitdepth > 8 ? bitdepth - 8 : 0;
    t.fixed_ok = t.n <= kMaxFixedTaps;
    for (int k = 0; k < t.n; ++k)
        if (t.t[k] != t.t[t.n - 1 - k])
            t.fixed_ok = 0;
    for (int k = 0; k < kMaxFixedTaps; ++k) {
        const float a = k < t.n ? std::ldexp(t.t[k], -q) : 0.0f;
        const float b = k < t.n ? std::ldexp(t.t[k], -2 * q) : 0.0f;
        if (k < t.n && (!(std::fabs(a) >= FLT_MIN) || !(std::fabs(b) >= FLT_MIN)))
            t.fixed_ok = 0;
        t.ra2[k] = make_float2(a, a);
        t.rb2[k] = make_float2(b, b);
        t.rc[k] = b;
    }
}

/* Constants of the per-pixel statistic.  nsq_up makes the fp64 comparison
 * (double)s1 < nsq an fp32 one: for an fp32 s1, s1 < nsq exactly when s1 is
 * below the smallest fp32 value not below nsq.  n_hi + n_lo carries nsq to
 * 2^-48 for the pair evaluation, which is used only for nsq in
 * [2^-60, 2^60] so that every pair quantity stays a normal fp32 value.    */
void make_term_params(double nsq, float gain_limit, int mode, TermParams &t)
{
    std::memset(&t, 0, sizeof t);
    t.nsq = nsq;
    t.gain_limit = gain_limit;
    t.one2 = make_float2(1.0f, 1.0f);
    float up = (float)nsq;
    if ((double)up < nsq)
        up = std::nextafter(up, INFINITY);
    t.nsq_up = up;
    const bool in_range = nsq >= 0x1p-60 && nsq <= 0x1p60;
    t.mode = in_range ? mode : kTermsFp64;
    if (in_range) {
        t.n_hi = (float)nsq;
        t.n_lo = (float)(nsq - (double)t.n_hi);
        t.rcp_n = (float)(1.0 / (double)t.n_hi);
        int e = 0;
        const double m = std::frexp(nsq, &e); /* nsq = m 2^e, m in [0.5, 1) */
        t.inv_pow2 = (m == 0.5) ? (float)std::ldexp(1.0, 1 - e) : 0.0f;
    }
}

} // namespace fvif

namespace {

/* Keeps the caller's current device; switches to the context's for the
 * duration of one API call. */
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess)
            return;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
            cudaSetDevice(prev);
    }
};

} // namespace

struct fvif_ctx {
    int w = 0, h = 0, bitdepth = 8;
    float kernelscale = 1.0f;
    double nsq = 2.0;
    float gain_limit = 100.0f;
    int skip_scale0 = 0;
    double min_val[kScales] = {0.0, 0.0, 0.0, 0.0};
    TermParams terms;
    int ws[kScales] = {}, hs[kScales] = {};
    Taps taps[kScales];
    int chunk = kDefaultChunk;
    /* frames per chunk of the host-input path (staging slot size): at most
     * kDefaultChunk, which measured fastest there (finer copy/score
     * interleaving), whatever the device-input chunk */
    int host_chunk = kDefaultChunk;
    /* test hook (FVIF_FAIL_ALLOC=n): allocation number n of this context
     * (0 = the first) fails as if the device were out of memory */
    int fail_alloc_at = -1;
    int allocs = 0;
    /* test hook (FVIF_TEST_DEC_STALL=1): the staged decimation's waits of
     * this context never complete, so each CTA gives up after its limit */
    unsigned dec_extra_tx = 0;
    int device = 0;
    cudaStream_t stream = nullptr;
    int last_status = FVIF_OK;

    /* Consecutive chunks alternate between two lanes, each with its own
     * stream and buffers, so one chunk's small kernels overlap the next
     * chunk's work.  Lanes fork from and join back into `stream`. */
    struct Lane {
        float2 *pyr[kScales] = {}; /* scales 1..3, chunk frames each      */
        float2 *rows = nullptr;    /* chunk frames x sum(h_s) (num, den)  */
        cudaStream_t stream = nullptr; /* low priority                     */
        cudaEvent_t done = nullptr;
        cudaEvent_t free_ev = nullptr; /* lane work before this chunk done */
        cudaEvent_t s0_done = nullptr; /* this chunk's scale-0 statistic   */
    } lanes[kLanes];
    /* Every scale-0 statistic launch runs on this one high-priority stream,
     * one chunk after the other: each gets the GPU to itself, and the
     * lanes' smaller kernels (low priority) fill the SMs it leaves idle. */
    cudaStream_t big = nullptr;
    cudaEvent_t fork = nullptr;
    int rows_stride = 0;
    int rows_base[kScales] = {};
    float2 *sums = nullptr;      /* chunk x 4 (diagnostics)               */

    /* bit 0 set by a decimation whose staged source tile did not arrive
     * within its wait limit; read and cleared by the synchronous calls   */
    unsigned *d_status = nullptr;
    unsigned *h_status = nullptr; /* pinned copy of d_status             */
    double *d_out = nullptr;     /* results of the synchronous calls      */
    double *h_out = nullptr;     /* pinned staging of d_out               */
    int out_cap = 0;
    float2 *d_sums = nullptr;    /* per-(frame, scale) sums (debug)       */
    double *d_debug = nullptr;   /* fifteen debug values per frame        */
    double *h_debug = nullptr;   /* pinned staging of d_debug             */
    int debug_cap = 0;

    /* opt-in launch timing: event pairs per kernel kind */
    bool profiling = false;
    std::vector<cudaEvent_t> prof_events[FVIF_K_COUNT];
    size_t prof_used[FVIF_K_COUNT] = {};
    long long launches[FVIF_K_COUNT] = {};

    /* host-input pipeline (allocated on first fvif_score_host) */
    int stage_slots = 3;        /* staging slots of the host path        */
    int host_lanes = kLanes;    /* compute lanes the host path uses      */
    unsigned char *stage[kMaxStage] = {};
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t copied[kMaxStage] = {};
    cudaEvent_t consumed[kMaxStage] = {};

    /* per-chunk timing of the last fvif_score_host call made while
     * profiling: the copy of each chunk on the copy stream, its scoring on
     * its lane (from the moment the lane may start it to the end of its
     * reduction), and the host time spent enqueueing it */
    struct HostChunk {
        cudaEvent_t copy0 = nullptr, copy1 = nullptr;
        cudaEvent_t score0 = nullptr, score1 = nullptr;
        double enq0 = 0.0, enq1 = 0.0; /* host ms since the call began */
        double locked = 0.0; /* 1: both input ranges page-locked       */
    };
    std::vector<HostChunk> host_prof;
    int host_prof_n = 0;

    size_t sample_bytes() const { return bitdepth == 8 ? 1u : 2u; }
    size_t frame_stride = 0; /* samples between consecutive input frames */
    size_t plane_bytes() const { return (size_t)w * h * sample_bytes(); }
    size_t frame_bytes() const { return frame_stride * sample_bytes(); }
};

namespace {

int set_status(fvif_ctx *ctx, int st)
{
    if (ctx)
        ctx->last_status = st;
    return st;
}

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess)
        return FVIF_OK;
    if (e == cudaErrorMemoryAllocation)
        return FVIF_ENOMEM;
    return FVIF_ECUDA;
}

/* Every device or pinned-host allocation of a context goes through these,
 * so the allocation-failure hook can fail any one of them. */
cudaError_t ctx_malloc(fvif_ctx *c, void **p, size_t n)
{
    if (c->allocs++ == c->fail_alloc_at)
        return cudaErrorMemoryAllocation;
    return cudaMalloc(p, n);
}

cudaError_t ctx_malloc_host(fvif_ctx *c, void **p, size_t n)
{
    if (c->allocs++ == c->fail_alloc_at)
        return cudaErrorMemoryAllocation;
    return cudaMallocHost(p, n);
}

/* The host-input pipeline (staging slots, their events, the copy stream);
 * leaves the context as if no pipeline had been made. */
void release_pipeline(fvif_ctx *c)
{
    for (int i = 0; i < kMaxStage; ++i) {
        if (c->stage[i])
            cudaFree(c->stage[i]);
        if (c->copied[i])
            cudaEventDestroy(c->copied[i]);
        if (c->consumed[i])
            cudaEventDestroy(c->consumed[i]);
        c->stage[i] = nullptr;
        c->copied[i] = nullptr;
        c->consumed[i] = nullptr;
    }
    if (c->copy_stream)
        cudaStreamDestroy(c->copy_stream);
    c->copy_stream = nullptr;
}

void release(fvif_ctx *c)
{
    for (fvif_ctx::Lane &l : c->lanes) {
        for (int s = 0; s < kScales; ++s)
            if (l.pyr[s])
                cudaFree(l.pyr[s]);
        if (l.rows)
            cudaFree(l.rows);
        if (l.stream)
            cudaStreamDestroy(l.stream);
        if (l.done)
            cudaEventDestroy(l.done);
        if (l.free_ev)
            cudaEventDestroy(l.free_ev);
        if (l.s0_done)
            cudaEventDestroy(l.s0_done);
    }
    if (c->big)
        cudaStreamDestroy(c->big);
    if (c->fork)
        cudaEventDestroy(c->fork);
    if (c->sums)
        cudaFree(c->sums);
    if (c->d_status)
        cudaFree(c->d_status);
    if (c->h_status)
        cudaFreeHost(c->h_status);
    if (c->d_out)
        cudaFree(c->d_out);
    if (c->h_out)
        cudaFreeHost(c->h_out);
    if (c->d_sums)
        cudaFree(c->d_sums);
    if (c->d_debug)
        cudaFree(c->d_debug);
    if (c->h_debug)
        cudaFreeHost(c->h_debug);
    release_pipeline(c);
    for (int k = 0; k < FVIF_K_COUNT; ++k)
        for (cudaEvent_t ev : c->prof_events[k])
            cudaEventDestroy(ev);
    for (fvif_ctx::HostChunk &h : c->host_prof)
        for (cudaEvent_t ev : {h.copy0, h.copy1, h.score0, h.score1})
            if (ev)
                cudaEventDestroy(ev);
}

/* The timing events of host-path chunk i, made on first use. */
cudaError_t host_chunk_events(fvif_ctx *c, int i, fvif_ctx::HostChunk **out)
{
    while ((int)c->host_prof.size() <= i) {
        fvif_ctx::HostChunk h;
        cudaError_t e = cudaSuccess;
        for (cudaEvent_t *ev : {&h.copy0, &h.copy1, &h.score0, &h.score1})
            if (e == cudaSuccess)
                e = cudaEventCreate(ev);
        if (e != cudaSuccess) {
            for (cudaEvent_t ev : {h.copy0, h.copy1, h.score0, h.score1})
                if (ev)
                    cudaEventDestroy(ev);
            return e;
        }
        c->host_prof.push_back(h);
    }
    *out = &c->host_prof[i];
    return cudaSuccess;
}

/* Record the start event of one launch of kind k (profiling only). */
cudaError_t prof_begin(fvif_ctx *c, int k, cudaStream_t st)
{
    c->launches[k] += 1;
    if (!c->profiling)
        return cudaSuccess;
    std::vector<cudaEvent_t> &v = c->prof_events[k];
    if (c->prof_used[k] + 2 > v.size()) {
        for (int i = 0; i < 2; ++i) {
            cudaEvent_t ev;
            cudaError_t e = cudaEventCreate(&ev);
            if (e != cudaSuccess)
                return e;
            v.push_back(ev);
        }
    }
    return cudaEventRecord(v[c->prof_used[k]], st);
}

cudaError_t prof_end(fvif_ctx *c, int k, cudaStream_t st)
{
    if (!c->profiling)
        return cudaSuccess;
    cudaError_t e =
        cudaEventRecord(c->prof_events[k][c->prof_used[k] + 1], st);
    c->prof_used[k] += 2;
    return e;
}

SrcDesc scale0_src(const fvif_ctx *c, const void *ref, const void *dist,
                   size_t frame_elems)
{
    SrcDesc d;
    d.kind = c->bitdepth == 8 ? SrcKind::U8 : SrcKind::U16;
    d.x = ref;
    d.y = dist;
    d.scale = c->bitdepth == 8 ? 1.0f
                               : std::ldexp(1.0f, -(c->bitdepth - 8));
    d.frame_elems = frame_elems;
    return d;
}

SrcDesc pyr_src(const fvif_ctx *c, const fvif_ctx::Lane &l, int s)
{
    SrcDesc d;
    d.kind = SrcKind::F2;
    d.x = l.pyr[s];
    d.y = nullptr;
    d.scale = 1.0f;
    d.frame_elems = (size_t)c->ws[s] * c->hs[s];
    return d;
}

/* One chunk (nf <= chunk frames) on the context stream: the pyramid, the
 * four statistic launches and the final reduction into out (device). */
int run_chunk(fvif_ctx *c, fvif_ctx::Lane &l, const void *ref,
              const void *dist, int nf, double *out, float2 *sums,
              size_t in_frame_elems)
{
    cudaStream_t st = l.stream;
    const SrcDesc s0 = scale0_src(c, ref, dist, in_frame_elems);
    /* the scale-0 statistic of this chunk may start once everything queued
     * on the lane before it is done (its input copied, the chunk that used
     * the lane's buffers before it reduced) */
    cudaError_t e = cudaEventRecord(l.free_ev, st);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(c->big, l.free_ev, 0);

    for (int s = 1; s < kScales && e == cudaSuccess; ++s) {
        DecArgs d;
        d.src = (s == 1) ? s0 : pyr_src(c, l, s - 1);
        d.w = c->ws[s - 1];
        d.h = c->hs[s - 1];
        d.nframes = nf;
        d.dst = l.pyr[s];
        d.dst_frame_elems = (size_t)c->ws[s] * c->hs[s];
        d.status = c->d_status;
        d.extra_tx = c->dec_extra_tx;
        e = prof_begin(c, FVIF_K_DECIMATE, st);
        if (e == cudaSuccess)
            e = launch_decimate(d, c->taps[s], st);
        if (e == cudaSuccess)
            e = prof_end(c, FVIF_K_DECIMATE, st);
    }
    for (int s = 0; s < kScales && e == cudaSuccess; ++s) {
        if (s == 0 && c->skip_scale0)
            continue;
        StatsArgs a;
        a.src = (s == 0) ? s0 : pyr_src(c, l, s);
        a.w = c->ws[s];
        a.h = c->hs[s];
        a.nframes = nf;
        a.terms = c->terms;
        a.rows = l.rows;
        a.rows_stride = c->rows_stride;
        a.rows_base = c->rows_base[s];
        const int kind = s == 0 ? FVIF_K_STATS0 : FVIF_K_STATS123;
        cudaStream_t ks = s == 0 ? c->big : st;
        e = prof_begin(c, kind, ks);
        if (e == cudaSuccess)
            e = launch_stats(a, c->taps[s], ks);
        if (e == cudaSuccess)
            e = prof_end(c, kind, ks);
        if (e == cudaSuccess && s == 0)
            e = cudaEventRecord(l.s0_done, c->big);
    }
    /* the reduction reads the scale-0 row sums */
    if (e == cudaSuccess && !c->skip_scale0)
        e = cudaStreamWaitEvent(st, l.s0_done, 0);
    if (e == cudaSuccess) {
        FinalArgs f;
        f.rows = l.rows;
        f.rows_stride = c->rows_stride;
        for (int s = 0; s < kScales; ++s) {
            f.rows_base[s] = c->rows_base[s];
            f.h[s] = c->hs[s];
        }
        f.nframes = nf;
        f.out = out;
        f.sums = sums;
        f.skip_scale0 = c->skip_scale0;
        for (int s = 0; s < kScales; ++s)
            f.min_val[s] = c->min_val[s];
        e = prof_begin(c, FVIF_K_FINAL, st);
        if (e == cudaSuccess)
            e = launch_final(f, st);
        if (e == cudaSuccess)
            e = prof_end(c, FVIF_K_FINAL, st);
    }
    return cuda_status(e);
}

/* The lanes start after everything already queued on the context stream. */
cudaError_t fork_lanes(fvif_ctx *c)
{
    cudaError_t e = cudaEventRecord(c->fork, c->stream);
    for (int i = 0; i < kLanes && e == cudaSuccess; ++i)
        e = cudaStreamWaitEvent(c->lanes[i].stream, c->fork, 0);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(c->big, c->fork, 0);
    return e;
}

/* Work queued on the context stream afterwards waits for both lanes. */
cudaError_t join_lanes(fvif_ctx *c)
{
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < kLanes && e == cudaSuccess; ++i) {
        e = cudaEventRecord(c->lanes[i].done, c->lanes[i].stream);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(c->stream, c->lanes[i].done, 0);
    }
    return e;
}

int enqueue_all(fvif_ctx *c, const void *ref, const void *dist, int n,
                double *out, float2 *sums = nullptr)
{
    const size_t fb = c->frame_bytes();
    int st = cuda_status(fork_lanes(c));
    int i = 0;
    for (int f0 = 0; f0 < n && st == FVIF_OK; f0 += c->chunk, ++i) {
        const int nf = (n - f0 < c->chunk) ? n - f0 : c->chunk;
        st = run_chunk(c, c->lanes[i % kLanes],
                       static_cast<const unsigned char *>(ref) + fb * f0,
                       static_cast<const unsigned char *>(dist) + fb * f0, nf,
                       out + (size_t)kScales * f0,
                       sums ? sums + (size_t)kScales * f0 : nullptr,
                       c->frame_stride);
    }
    const int sj = cuda_status(join_lanes(c));
    return st != FVIF_OK ? st : sj;
}

int ensure_out(fvif_ctx *c, int n)
{
    if (n <= c->out_cap)
        return FVIF_OK;
    int cap = c->out_cap ? c->out_cap : 256;
    while (cap < n)
        cap *= 2;
    double *d = nullptr, *h = nullptr;
    if (ctx_malloc(c, (void **)&d, sizeof(double) * kScales * (size_t)cap) !=
        cudaSuccess)
        return FVIF_ENOMEM;
    if (ctx_malloc_host(c, (void **)&h,
                        sizeof(double) * kScales * (size_t)cap) !=
        cudaSuccess) {
        cudaFree(d);
        return FVIF_ENOMEM;
    }
    if (c->d_out)
        cudaFree(c->d_out);
    if (c->h_out)
        cudaFreeHost(c->h_out);
    c->d_out = d;
    c->h_out = h;
    c->out_cap = cap;
    return FVIF_OK;
}

int ensure_debug(fvif_ctx *c, int n)
{
    if (n <= c->debug_cap)
        return FVIF_OK;
    int cap = c->debug_cap ? c->debug_cap : 64;
    while (cap < n)
        cap *= 2;
    float2 *sm = nullptr;
    double *d = nullptr, *h = nullptr;
    cudaError_t e = ctx_malloc(c, (void **)&sm,
                               sizeof(float2) * kScales * (size_t)cap);
    if (e == cudaSuccess)
        e = ctx_malloc(c, (void **)&d, sizeof(double) * 15 * (size_t)cap);
    if (e == cudaSuccess)
        e = ctx_malloc_host(c, (void **)&h,
                            sizeof(double) * 15 * (size_t)cap);
    if (e != cudaSuccess) {
        if (sm)
            cudaFree(sm);
        if (d)
            cudaFree(d);
        return FVIF_ENOMEM;
    }
    if (c->d_sums)
        cudaFree(c->d_sums);
    if (c->d_debug)
        cudaFree(c->d_debug);
    if (c->h_debug)
        cudaFreeHost(c->h_debug);
    c->d_sums = sm;
    c->d_debug = d;
    c->h_debug = h;
    c->debug_cap = cap;
    return FVIF_OK;
}

/* Enqueue the read of the context's device status word (after the work
 * queued on the context stream). */
cudaError_t status_to_host(fvif_ctx *c)
{
    return cudaMemcpyAsync(c->h_status, c->d_status, sizeof(unsigned),
                           cudaMemcpyDeviceToHost, c->stream);
}

/* After the stream is synchronised: FVIF_ECUDA if a kernel marked the
 * status word (which is then cleared for the next call), else FVIF_OK. */
int status_check(fvif_ctx *c)
{
    if (*c->h_status == 0)
        return FVIF_OK;
    *c->h_status = 0;
    cudaMemsetAsync(c->d_status, 0, sizeof(unsigned), c->stream);
    cudaStreamSynchronize(c->stream);
    return FVIF_ECUDA;
}

int finish_to_host(fvif_ctx *c, int n, double *out)
{
    cudaError_t e = cudaMemcpyAsync(c->h_out, c->d_out,
                                    sizeof(double) * kScales * (size_t)n,
                                    cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess)
        e = status_to_host(c);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess)
        return cuda_status(e);
    const int st = status_check(c);
    if (st != FVIF_OK)
        return st;
    std::memcpy(out, c->h_out, sizeof(double) * kScales * (size_t)n);
    return FVIF_OK;
}

int ensure_pipeline(fvif_ctx *c)
{
    if (c->copy_stream)
        return FVIF_OK;
    const size_t slot = 2 * c->plane_bytes() * (size_t)c->host_chunk;
    cudaError_t e = cudaStreamCreateWithFlags(&c->copy_stream,
                                              cudaStreamNonBlocking);
    for (int i = 0; i < c->stage_slots && e == cudaSuccess; ++i) {
        e = ctx_malloc(c, (void **)&c->stage[i], slot);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&c->copied[i],
                                         cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&c->consumed[i],
                                         cudaEventDisableTiming);
    }
    /* a pipeline that could not be made completely is not kept: the next
     * call tries again instead of using missing slots */
    if (e != cudaSuccess)
        release_pipeline(c);
    return cuda_status(e);
}

/* FVIF_LOG set (to anything) in the environment: one line on stderr per
 * create and score call, with its size, status and host wall time. */
bool log_enabled()
{
    static const bool on = std::getenv("FVIF_LOG") != nullptr;
    return on;
}

double ms_since(std::chrono::steady_clock::time_point t0)
{
    return std::chrono::duration<double, std::milli>(
               std::chrono::steady_clock::now() - t0)
        .count();
}

void log_call(const char *what, const fvif_ctx *c, int n_frames, int st,
              std::chrono::steady_clock::time_point t0)
{
    if (!log_enabled())
        return;
    if (!live(c))
        c = nullptr;     /* a stray pointer is reported, not read */
    std::fprintf(stderr,
                 "fvif: %s %dx%d frames=%d chunk=%d status=%d (%s) "
                 "%.3f ms\n",
                 what, c ? c->w : 0, c ? c->h : 0, n_frames,
                 c ? c->chunk : 0, st, fvif_strerror(st), ms_since(t0));
}

} // namespace

extern "C" {

void fvif_default_options(fvif_options *opt)
{
    if (!opt)
        return;
    opt->enhn_gain_limit = 100.0f;
    opt->skip_scale0 = 0;
    opt->frame_stride = 0;
    for (int s = 0; s < kScales; ++s)
        opt->min_val[s] = 0.0;
}

fvif_ctx *fvif_create(int w, int h, int bitdepth, float kernelscale,
                      double sigma_nsq)
{
    return fvif_create_ex(w, h, bitdepth, kernelscale, sigma_nsq, nullptr);
}

static fvif_ctx *create_ex_impl(int w, int h, int bitdepth, float kernelscale,
                         double sigma_nsq, const fvif_options *opt)
{
    g_create_status = FVIF_EINVAL;
    fvif_options o;
    fvif_default_options(&o);
    if (opt)
        o = *opt;
    if (!(o.enhn_gain_limit > 0.0f) || !std::isfinite(o.enhn_gain_limit))
        return nullptr;
    for (int s = 0; s < kScales; ++s)
        if (!std::isfinite(o.min_val[s]))
            return nullptr;
    if (o.frame_stride != 0 && o.frame_stride < (long long)w * h)
        return nullptr;
    if (w < 16 || h < 16 || w > 16384 || h > 16384)
        return nullptr;
    if (bitdepth < 8 || bitdepth > 16)
        return nullptr;
    if (!(kernelscale > 0.0f) || !std::isfinite(kernelscale))
        return nullptr;
    if (!(sigma_nsq > 0.0) || !std::isfinite(sigma_nsq))
        return nullptr;

    fvif_ctx *c = new (std::nothrow) fvif_ctx();
    if (!c) {
        g_create_status = FVIF_ENOMEM;
        return nullptr;
    }
    c->w = w;
    c->h = h;
    c->bitdepth = bitdepth;
    c->kernelscale = kernelscale;
    c->nsq = sigma_nsq;
    c->frame_stride = o.frame_stride ? (size_t)o.frame_stride
                                     : (size_t)w * (size_t)h;
    c->gain_limit = o.enhn_gain_limit;
    c->skip_scale0 = o.skip_scale0 ? 1 : 0;
    for (int s = 1; s < kScales; ++s)
        c->min_val[s] = o.min_val[s];
    {
        const char *mode = std::getenv("FVIF_TERMS");
        const int m = (mode && std::strcmp(mode, "fp64") == 0) ? kTermsFp64
                                                               : kTermsPair;
        make_term_params(sigma_nsq, c->gain_limit, m, c->terms);
    }
    for (int s = 0; s < kScales; ++s) {
        c->ws[s] = s == 0 ? w : c->ws[s - 1] / 2;
        c->hs[s] = s == 0 ? h : c->hs[s - 1] / 2;
        if (make_taps(kernelscale, s, c->taps[s]) != FVIF_OK) {
            delete c;
            return nullptr;
        }
        set_sample_taps(c->taps[s], bitdepth);
    }
    /* Frames per chunk: enough that the scale-0 statistic launch has about
     * kChunkCtas CTAs (one per 16-row strip and frame; measured best for
     * 576x324, 1080p and 4K alike), at least kDefaultChunk frames. */
    {
        const int strips = (h + 15) / 16;
        int v = (kChunkCtas + strips - 1) / strips;
        v = v < kDefaultChunk ? kDefaultChunk : (v > kMaxChunk ? kMaxChunk : v);
        c->chunk = v;
    }
    if (const char *env = std::getenv("FVIF_CHUNK")) {
        const int v = std::atoi(env);
        if (v > 0 && v <= kMaxChunk)
            c->chunk = v;
    }
    c->host_chunk = c->chunk < kDefaultChunk ? c->chunk : kDefaultChunk;
    if (const char *env = std::getenv("FVIF_FAIL_ALLOC")) {
        char *end = nullptr;
        const long v = std::strtol(env, &end, 10);
        if (end != env && v >= 0 && v < 1000000)
            c->fail_alloc_at = (int)v;
    }
    if (const char *env = std::getenv("FVIF_HOST_SLOTS")) {
        const int v = std::atoi(env);
        if (v >= 2 && v <= kMaxStage)
            c->stage_slots = v;
    }
    if (const char *env = std::getenv("FVIF_TEST_DEC_STALL"))
        c->dec_extra_tx = std::atoi(env) != 0 ? 16u : 0u;
    if (const char *env = std::getenv("FVIF_HOST_LANES")) {
        const int v = std::atoi(env);
        if (v >= 1 && v <= kLanes)
            c->host_lanes = v;
    }
    cudaError_t e = cudaGetDevice(&c->device);
    int prio_low = 0, prio_high = 0;
    if (e == cudaSuccess)
        e = cudaDeviceGetStreamPriorityRange(&prio_low, &prio_high);
    int rows_total = 0;
    for (int s = 0; s < kScales; ++s) {
        c->rows_base[s] = rows_total;
        rows_total += c->hs[s];
    }
    c->rows_stride = rows_total;
    for (int i = 0; i < kLanes && e == cudaSuccess; ++i) {
        fvif_ctx::Lane &l = c->lanes[i];
        for (int s = 1; s < kScales && e == cudaSuccess; ++s)
            e = ctx_malloc(c, (void **)&l.pyr[s],
                           sizeof(float2) * (size_t)c->ws[s] * c->hs[s] *
                               c->chunk);
        if (e == cudaSuccess)
            e = ctx_malloc(c, (void **)&l.rows,
                           sizeof(float2) * (size_t)rows_total * c->chunk);
        if (e == cudaSuccess)
            e = cudaStreamCreateWithPriority(&l.stream, cudaStreamNonBlocking,
                                             prio_low);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&l.done, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&l.free_ev, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&l.s0_done, cudaEventDisableTiming);
    }
    if (e == cudaSuccess)
        e = cudaStreamCreateWithPriority(&c->big, cudaStreamNonBlocking,
                                         prio_high);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&c->fork, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = ctx_malloc(c, (void **)&c->sums,
                       sizeof(float2) * kScales * (size_t)c->chunk);
    if (e == cudaSuccess)
        e = ctx_malloc(c, (void **)&c->d_status, sizeof(unsigned));
    if (e == cudaSuccess)
        e = ctx_malloc_host(c, (void **)&c->h_status, sizeof(unsigned));
    if (e == cudaSuccess) {
        *c->h_status = 0;
        e = cudaMemset(c->d_status, 0, sizeof(unsigned));
    }
    int st = cuda_status(e);
    if (st == FVIF_OK)
        st = ensure_out(c, c->chunk);
    if (st != FVIF_OK) {
        release(c);
        delete c;
        g_create_status = st;
        return nullptr;
    }
    g_create_status = FVIF_OK;
    return c;
}

void fvif_destroy(fvif_ctx *ctx)
{
    {
        std::lock_guard<std::mutex> lock(g_live_mutex);
        if (!ctx || g_live.erase(ctx) == 0)
            return;
    }
    DeviceGuard g(ctx->device);
    cudaStreamSynchronize(ctx->stream);
    for (fvif_ctx::Lane &l : ctx->lanes)
        if (l.stream)
            cudaStreamSynchronize(l.stream);
    release(ctx);
    delete ctx;
}

int fvif_set_stream(fvif_ctx *ctx, void *cuda_stream)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    ctx->stream = static_cast<cudaStream_t>(cuda_stream);
    return set_status(ctx, FVIF_OK);
}

int fvif_last_error(const fvif_ctx *ctx)
{
    if (!ctx)
        return g_create_status;
    return live(ctx) ? ctx->last_status : FVIF_EINVAL;
}

const char *fvif_strerror(int status)
{
    switch (status) {
    case FVIF_OK: return "ok";
    case FVIF_EINVAL: return "invalid argument";
    case FVIF_ENOMEM: return "out of memory";
    case FVIF_ECUDA: return "CUDA error";
    case FVIF_ETOOBIG:
        return "frame too large for the no-allocation entry point's scratch";
    default: return "unknown status";
    }
}

int fvif_profile_enable(fvif_ctx *ctx, int enable)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    DeviceGuard g(ctx->device);
    if (cudaStreamSynchronize(ctx->stream) != cudaSuccess)
        return set_status(ctx, FVIF_ECUDA);
    for (fvif_ctx::Lane &l : ctx->lanes)
        if (cudaStreamSynchronize(l.stream) != cudaSuccess)
            return set_status(ctx, FVIF_ECUDA);
    ctx->profiling = enable != 0;
    for (int k = 0; k < FVIF_K_COUNT; ++k) {
        ctx->prof_used[k] = 0;
        ctx->launches[k] = 0;
    }
    return set_status(ctx, FVIF_OK);
}

int fvif_profile_read(fvif_ctx *ctx, int kind, double *total_ms,
                      long long *launches)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    if (kind < 0 || kind >= FVIF_K_COUNT || !total_ms || !launches)
        return set_status(ctx, FVIF_EINVAL);
    DeviceGuard g(ctx->device);
    double ms = 0.0;
    const std::vector<cudaEvent_t> &v = ctx->prof_events[kind];
    for (size_t i = 0; i + 1 < ctx->prof_used[kind]; i += 2) {
        if (cudaEventSynchronize(v[i + 1]) != cudaSuccess)
            return set_status(ctx, FVIF_ECUDA);
        float t = 0.0f;
        if (cudaEventElapsedTime(&t, v[i], v[i + 1]) != cudaSuccess)
            return set_status(ctx, FVIF_ECUDA);
        ms += t;
    }
    *total_ms = ms;
    *launches = ctx->launches[kind];
    return set_status(ctx, FVIF_OK);
}

int fvif_profile_host(fvif_ctx *ctx, double *out, int cap)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    if (cap < 0 || (cap > 0 && !out))
        return set_status(ctx, FVIF_EINVAL);
    DeviceGuard g(ctx->device);
    if (!g.ok)
        return set_status(ctx, FVIF_ECUDA);
    const int n = ctx->host_prof_n;
    for (int i = 0; i < n && i < cap; ++i) {
        const fvif_ctx::HostChunk &h = ctx->host_prof[i];
        const cudaEvent_t evs[4] = {h.copy0, h.copy1, h.score0, h.score1};
        for (int k = 0; k < 4; ++k) {
            float t = 0.0f;
            cudaError_t e = cudaEventSynchronize(evs[k]);
            if (e == cudaSuccess)
                e = cudaEventElapsedTime(&t, ctx->host_prof[0].copy0, evs[k]);
            if (e != cudaSuccess)
                return set_status(ctx, cuda_status(e));
            out[7 * i + k] = t;
        }
        out[7 * i + 4] = h.enq0;
        out[7 * i + 5] = h.enq1;
        out[7 * i + 6] = h.locked;
    }
    set_status(ctx, FVIF_OK);
    return n;
}

int fvif_chunk_frames(const fvif_ctx *ctx)
{
    return live(ctx) ? ctx->chunk : FVIF_EINVAL;
}

int fvif_get_taps(const fvif_ctx *ctx, int scale, float *taps, int cap)
{
    if (!live(ctx) || !taps || scale < 0 || scale >= kScales)
        return FVIF_EINVAL;
    const Taps &t = ctx->taps[scale];
    if (cap < t.n)
        return FVIF_EINVAL;
    std::memcpy(taps, t.t, sizeof(float) * t.n);
    return t.n;
}

static int score_async_impl(fvif_ctx *ctx, const void *ref, const void *dist,
                     int n_frames, double *out)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    if (n_frames < 0 || (n_frames > 0 && (!ref || !dist || !out)))
        return set_status(ctx, FVIF_EINVAL);
    if (n_frames == 0)
        return set_status(ctx, FVIF_OK);
    DeviceGuard g(ctx->device);
    if (!g.ok)
        return set_status(ctx, FVIF_ECUDA);
    return set_status(ctx, enqueue_all(ctx, ref, dist, n_frames, out));
}

static int score_impl(fvif_ctx *ctx, const void *ref, const void *dist, int n_frames,
               double *out)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    if (n_frames < 0 || (n_frames > 0 && (!ref || !dist || !out)))
        return set_status(ctx, FVIF_EINVAL);
    if (n_frames == 0)
        return set_status(ctx, FVIF_OK);
    DeviceGuard g(ctx->device);
    if (!g.ok)
        return set_status(ctx, FVIF_ECUDA);
    int st = ensure_out(ctx, n_frames);
    if (st == FVIF_OK)
        st = enqueue_all(ctx, ref, dist, n_frames, ctx->d_out);
    if (st == FVIF_OK)
        st = finish_to_host(ctx, n_frames, out);
    return set_status(ctx, st);
}

static int score_debug_impl(fvif_ctx *ctx, const void *ref, const void *dist,
                     int n_frames, double *out)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    if (n_frames < 0 || (n_frames > 0 && (!ref || !dist || !out)))
        return set_status(ctx, FVIF_EINVAL);
    if (n_frames == 0)
        return set_status(ctx, FVIF_OK);
    DeviceGuard g(ctx->device);
    if (!g.ok)
        return set_status(ctx, FVIF_ECUDA);
    int st = ensure_out(ctx, n_frames);
    if (st == FVIF_OK)
        st = ensure_debug(ctx, n_frames);
    if (st == FVIF_OK)
        st = enqueue_all(ctx, ref, dist, n_frames, ctx->d_out, ctx->d_sums);
    if (st == FVIF_OK)
        st = cuda_status(launch_debug(ctx->d_out, ctx->d_sums, n_frames,
                                      ctx->d_debug, ctx->stream));
    cudaError_t e = cudaSuccess;
    if (st == FVIF_OK)
        e = cudaMemcpyAsync(ctx->h_debug, ctx->d_debug,
                            sizeof(double) * 15 * (size_t)n_frames,
                            cudaMemcpyDeviceToHost, ctx->stream);
    if (st == FVIF_OK && e == cudaSuccess)
        e = status_to_host(ctx);
    if (st == FVIF_OK && e == cudaSuccess)
        e = cudaStreamSynchronize(ctx->stream);
    if (st == FVIF_OK && e != cudaSuccess)
        st = cuda_status(e);
    if (st == FVIF_OK)
        st = status_check(ctx);
    if (st == FVIF_OK)
        std::memcpy(out, ctx->h_debug, sizeof(double) * 15 * (size_t)n_frames);
    return set_status(ctx, st);
}

/* Whether host range [p, p + n) is page-locked (allocated by
 * cudaHostAlloc / cudaMallocHost or registered with cudaHostRegister), as
 * this process's CUDA runtime sees it: both ends are checked.  Clears the
 * error a pageable pointer leaves behind on older runtimes. */
static bool page_locked(const void *p, size_t n)
{
    for (const unsigned char *q :
         {static_cast<const unsigned char *>(p),
          static_cast<const unsigned char *>(p) + (n ? n - 1 : 0)}) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (a.type != cudaMemoryTypeHost)
            return false;
    }
    return true;
}

static int score_host_impl(fvif_ctx *ctx, const void *ref, const void *dist,
                    int n_frames, double *out)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    if (n_frames < 0 || (n_frames > 0 && (!ref || !dist || !out)))
        return set_status(ctx, FVIF_EINVAL);
    if (n_frames == 0)
        return set_status(ctx, FVIF_OK);
    DeviceGuard g(ctx->device);
    if (!g.ok)
        return set_status(ctx, FVIF_ECUDA);
    int st = ensure_out(ctx, n_frames);
    if (st == FVIF_OK)
        st = ensure_pipeline(ctx);
    if (st != FVIF_OK)
        return set_status(ctx, st);

    /* the staging slots hold the luma planes packed (w*h samples apart);
     * the host frames may be further apart (frame_stride) */
    const size_t fb = ctx->frame_bytes();
    const size_t pb = ctx->plane_bytes();
    const int hc = ctx->host_chunk;
    const size_t half = pb * (size_t)hc;
    const bool prof = ctx->profiling;
    const auto t_call = std::chrono::steady_clock::now();
    if (prof)
        ctx->host_prof_n = 0;
    cudaError_t e = fork_lanes(ctx);
    /* The first chunk is a quarter chunk: scoring starts once it has been
     * copied instead of waiting for a whole chunk to cross the host link. */
    const int first = hc >= 4 ? hc / 4 : hc;
    int i = 0;
    for (int f0 = 0, nf = 0; f0 < n_frames && e == cudaSuccess;
         f0 += nf, ++i) {
        const int want = i == 0 ? first : hc;
        nf = (n_frames - f0 < want) ? n_frames - f0 : want;
        /* chunk i is copied into staging slot i % slots while earlier
         * chunks are scored, and scored on lane i % lanes */
        const int slot = i % ctx->stage_slots;
        fvif_ctx::Lane &lane = ctx->lanes[i % ctx->host_lanes];
        unsigned char *dref = ctx->stage[slot];
        unsigned char *ddist = ctx->stage[slot] + half;
        fvif_ctx::HostChunk *hp = nullptr;
        if (prof) {
            e = host_chunk_events(ctx, i, &hp);
            if (e != cudaSuccess)
                break;
            hp->enq0 = ms_since(t_call);
        }
        const unsigned char *href =
            static_cast<const unsigned char *>(ref) + fb * f0;
        const unsigned char *hdist =
            static_cast<const unsigned char *>(dist) + fb * f0;
        if (prof)
            hp->locked = page_locked(href, fb * (nf - 1) + pb) &&
                                 page_locked(hdist, fb * (nf - 1) + pb)
                             ? 1.0
                             : 0.0;
        /* the slot is free once the chunk that used it last was scored */
        e = cudaStreamWaitEvent(ctx->copy_stream, ctx->consumed[slot], 0);
        if (e == cudaSuccess && prof)
            e = cudaEventRecord(hp->copy0, ctx->copy_stream);
        /* packed luma planes: one plain copy per plane set; planes further
         * apart (planar YUV frames): one 2-D copy that skips the chroma */
        if (e == cudaSuccess)
            e = fb == pb ? cudaMemcpyAsync(dref, href, pb * nf,
                                           cudaMemcpyHostToDevice,
                                           ctx->copy_stream)
                         : cudaMemcpy2DAsync(dref, pb, href, fb, pb, nf,
                                             cudaMemcpyHostToDevice,
                                             ctx->copy_stream);
        if (e == cudaSuccess)
            e = fb == pb ? cudaMemcpyAsync(ddist, hdist, pb * nf,
                                           cudaMemcpyHostToDevice,
                                           ctx->copy_stream)
                         : cudaMemcpy2DAsync(ddist, pb, hdist, fb, pb, nf,
                                             cudaMemcpyHostToDevice,
                                             ctx->copy_stream);
        if (e == cudaSuccess && prof)
            e = cudaEventRecord(hp->copy1, ctx->copy_stream);
        if (e == cudaSuccess)
            e = cudaEventRecord(ctx->copied[slot], ctx->copy_stream);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(lane.stream, ctx->copied[slot], 0);
        if (e == cudaSuccess && prof)
            e = cudaEventRecord(hp->score0, lane.stream);
        if (e != cudaSuccess)
            break;
        st = run_chunk(ctx, lane, dref, ddist, nf,
                       ctx->d_out + (size_t)kScales * f0, nullptr,
                       (size_t)ctx->w * ctx->h);
        if (st != FVIF_OK)
            break;
        if (prof)
            e = cudaEventRecord(hp->score1, lane.stream);
        if (e == cudaSuccess)
            e = cudaEventRecord(ctx->consumed[slot], lane.stream);
        if (prof) {
            hp->enq1 = ms_since(t_call);
            ctx->host_prof_n = i + 1;
        }
    }
    const cudaError_t ej = join_lanes(ctx);
    if (e != cudaSuccess || st != FVIF_OK || ej != cudaSuccess) {
        cudaStreamSynchronize(ctx->copy_stream);
        cudaStreamSynchronize(ctx->stream);
        return set_status(ctx, st != FVIF_OK ? st
                               : cuda_status(e != cudaSuccess ? e : ej));
    }
    return set_status(ctx, finish_to_host(ctx, n_frames, out));
}

int fvif_debug_terms(fvif_ctx *ctx, const float *mu1, const float *mu2,
                     const float *xx, const float *yy, const float *xy,
                     int n, float *num, float *den,
                     unsigned long long *fallbacks)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    if (n < 0 || (n > 0 && (!mu1 || !mu2 || !xx || !yy || !xy || !num ||
                            !den)))
        return set_status(ctx, FVIF_EINVAL);
    if (n == 0)
        return set_status(ctx, FVIF_OK);
    DeviceGuard g(ctx->device);
    if (!g.ok)
        return set_status(ctx, FVIF_ECUDA);
    return set_status(ctx, cuda_status(launch_terms(ctx->terms, mu1, mu2, xx,
                                                    yy, xy, n, num, den,
                                                    fallbacks, ctx->stream)));
}

int fvif_debug_frame(fvif_ctx *ctx, const void *ref, const void *dist,
                     float *planes, float *rows, float *sums)
{
    if (!live(ctx))
        return FVIF_EINVAL;
    if (!ref || !dist)
        return set_status(ctx, FVIF_EINVAL);
    DeviceGuard g(ctx->device);
    if (!g.ok)
        return set_status(ctx, FVIF_ECUDA);
    fvif_ctx::Lane &lane = ctx->lanes[0];
    int st = cuda_status(fork_lanes(ctx));
    if (st == FVIF_OK)
        st = run_chunk(ctx, lane, ref, dist, 1, ctx->d_out, ctx->sums,
                       (size_t)ctx->w * ctx->h);
    const int sj = cuda_status(join_lanes(ctx));
    if (st == FVIF_OK)
        st = sj;
    if (st != FVIF_OK)
        return set_status(ctx, st);
    cudaError_t e = cudaSuccess;
    if (planes) {
        size_t total = 0;
        for (int s = 0; s < kScales; ++s)
            total += 2 * (size_t)ctx->ws[s] * ctx->hs[s];
        float *tmp = nullptr;
        e = ctx_malloc(ctx, (void **)&tmp, sizeof(float) * total);
        size_t off = 0;
        for (int s = 0; s < kScales && e == cudaSuccess; ++s) {
            const size_t np = (size_t)ctx->ws[s] * ctx->hs[s];
            const SrcDesc d =
                s == 0 ? scale0_src(ctx, ref, dist, (size_t)ctx->w * ctx->h)
                       : pyr_src(ctx, lane, s);
            e = launch_unpack_planes(d, ctx->ws[s], ctx->hs[s], tmp + off,
                                     tmp + off + np, ctx->stream);
            off += 2 * np;
        }
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(planes, tmp, sizeof(float) * total,
                                cudaMemcpyDeviceToHost, ctx->stream);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(ctx->stream);
        if (tmp)
            cudaFree(tmp);
        if (e != cudaSuccess)
            return set_status(ctx, cuda_status(e));
    }
    if (rows) {
        size_t off = 0;
        for (int s = 0; s < kScales && e == cudaSuccess; ++s) {
            e = cudaMemcpyAsync(rows + off, lane.rows + ctx->rows_base[s],
                                sizeof(float2) * ctx->hs[s],
                                cudaMemcpyDeviceToHost, ctx->stream);
            off += 2 * (size_t)ctx->hs[s];
        }
    }
    if (sums && e == cudaSuccess)
        e = cudaMemcpyAsync(sums, ctx->sums, sizeof(float2) * kScales,
                            cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(ctx->stream);
    return set_status(ctx, cuda_status(e));
}

fvif_ctx *fvif_create_ex(int w, int h, int bitdepth, float kernelscale,
                         double sigma_nsq, const fvif_options *opt)
{
    const auto t0 = std::chrono::steady_clock::now();
    fvif_ctx *c = create_ex_impl(w, h, bitdepth, kernelscale, sigma_nsq, opt);
    if (c) {
        std::lock_guard<std::mutex> lock(g_live_mutex);
        g_live.insert(c);
    }
    if (log_enabled())
        std::fprintf(stderr,
                     "fvif: create %dx%d bitdepth=%d kernelscale=%g "
                     "sigma_nsq=%g chunk=%d status=%d (%s) %.3f ms\n",
                     w, h, bitdepth, (double)kernelscale, sigma_nsq,
                     c ? c->chunk : 0, fvif_last_error(c),
                     fvif_strerror(fvif_last_error(c)), ms_since(t0));
    return c;
}

int fvif_score(fvif_ctx *ctx, const void *ref, const void *dist, int n_frames,
               double *out)
{
    const auto t0 = std::chrono::steady_clock::now();
    const int st = score_impl(ctx, ref, dist, n_frames, out);
    log_call("score", ctx, n_frames, st, t0);
    return st;
}

int fvif_score_async(fvif_ctx *ctx, const void *ref, const void *dist,
                     int n_frames, double *out)
{
    const auto t0 = std::chrono::steady_clock::now();
    const int st = score_async_impl(ctx, ref, dist, n_frames, out);
    log_call("score_async (enqueue)", ctx, n_frames, st, t0);
    return st;
}

int fvif_score_host(fvif_ctx *ctx, const void *ref, const void *dist,
                    int n_frames, double *out)
{
    const auto t0 = std::chrono::steady_clock::now();
    const int st = score_host_impl(ctx, ref, dist, n_frames, out);
    log_call("score_host", ctx, n_frames, st, t0);
    return st;
}

int fvif_score_debug(fvif_ctx *ctx, const void *ref, const void *dist,
                     int n_frames, double *out)
{
    const auto t0 = std::chrono::steady_clock::now();
    const int st = score_debug_impl(ctx, ref, dist, n_frames, out);
    log_call("score_debug", ctx, n_frames, st, t0);
    return st;
}

} // extern "C"
