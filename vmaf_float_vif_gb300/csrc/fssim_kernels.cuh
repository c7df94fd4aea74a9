/*
 * fssim_kernels.cuh -- kernels of float_ssim's auto-scale decimation.
 *
 * Source: "Research-2130: float_ssim decimation on the SYCL device" (Question:
 * the auto scale; Sources: the kernel, window offsets, boundary, sample
 * conversion and decimated size; Findings, "The CPU sum is exact").
 *
 * Each output is one fp32 rounding of the exact sum, over a k x k window
 * (k = scale, period-2n mirror at the edges), of the fp32 products
 * fl(x * t), x the converted sample and t = fl(1 / k^2).  With x = s * 2^-q
 * (s the integer sample, q = bitdepth - 8) and t = T * 2^-E (T a 24-bit
 * integer):
 *
 *   fl(x * t) = 2^-q * (s * t - e(s)),   e(s) = s * t - fl(s * t),
 *
 * where e(s) is exactly the FMA fma(s, t, -fl(s * t)) and an integer
 * multiple of 2^-E with |e| <= 2^15 * 2^-E.  So the window sum is
 *
 *   2^-(q + E) * (T * sum(s) - sum(e * 2^E))
 *
 * with both sums integers: sum(s) <= k^2 * 65535 < 2^31 and
 * |sum(e * 2^E)| <= k^2 * 2^15 <= 2^29 for k <= 128.  The int64 total is
 * rounded once to fp32 (__ll2float_rn), and the power-of-two factor is
 * applied exactly.  (The window kernel, k <= 7, forms the same rounding in
 * fp32 alone; see there.)  For power-of-two k the tap is exact: e = 0 and
 * the output is fl(sum(s)) * t * 2^-q.
 *
 * Three kernels, chosen per sample type and scale (measured at 4K):
 *  - ssim_decimate_u8_partials_kernel: 8-bit samples, k = 4 or 8, 16-byte
 *    rows: window partial sums with dp4a, no shared memory; at the HBM
 *    bound.
 *  - ssim_decimate_windows_kernel: k = 2..8, 16-byte rows: each thread owns
 *    16 (8-bit) or 8 (16-bit) whole windows; at k = 3 the block's rows are
 *    staged in shared memory by bulk asynchronous copies.
 *  - ssim_decimate_kernel, the general two-phase kernel, for every other
 *    case (any scale, any alignment).  A block takes R output rows by X
 *    output columns of one plane of one frame.  Phase 1: each thread sums V
 *    adjacent input columns (one 16-byte load per row on the vector path)
 *    over the k window rows of its output rows, into sum(s) as integers and
 *    sum(e) as fp32.  The fp32 sum is exact: each partial sum is a multiple
 *    of 2^-E below k * 2^15 * 2^-E < 2^24 * 2^-E.  The loads of a batch of
 *    rows are all issued before any is added.  The column sums go to shared
 *    memory as integers.  Phase 2: each thread adds the k columns of one
 *    output window, mirrored at the edges, and rounds once.
 * Every input byte is read from DRAM once (edge windows re-read mirrored
 * columns from shared memory or neighbouring lanes).  Exact taps are bound
 * by HBM bandwidth; inexact taps add about four instructions per sample for
 * the product error and are bound by instruction issue at 8 bits.
 *
 * The scales 2..8 (the auto scales of frames up to 8.5K wide) are compiled
 * with k fixed, so the row and column loops unroll; other scales run the
 * general kernel with k read at run time.
 */
#ifndef FSSIM_KERNELS_CUH
#define FSSIM_KERNELS_CUH

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace fssim {

constexpr int kThreads = 256;
constexpr int kMaxTileCols = 4096;          // window columns per tile row
constexpr int kMaxRows = 16;                // output rows per block
constexpr size_t kMaxSmem = 64 * 1024;      // shared bytes per block
constexpr int kMaxFramesPerLaunch = 32767;  // grid.z = 2 * frames
constexpr int kBatch = 8;                   // rows loaded before any is added

struct DecimateParams {
    const void *src[2];       // ref, dist
    float *dst[2];
    size_t in_frame_elems;
    size_t out_frame_elems;
    int w, h, k, sw, sh;
    int X, R;                 // outputs per tile row, output rows per block
    int pitch;                // shared row pitch in ints (skewed)
    float tap;                // fl(1 / k^2)
    float err_scale;          // 2^E: e * 2^E is an integer
    long long T;              // tap = T * 2^-E
    float out_scale;          // 2^-(q + E), or tap * 2^-q for exact taps
    int packed16;             // 16-bit samples: column sums fit 16 bits
    float2 one2;              // (1, 1)
    float inv_q;              // 2^-q
    unsigned stage_extra_tx;  // bytes the staged kernel waits for in excess
                              // of its copies (0; tests only)
};

/* Period-2n symmetric mirror: -1 -> 0, n -> n - 1, repeating with period 2n. */
__device__ __forceinline__ int mirror2n(int j, int n)
{
    if (j >= 0 && j < n)
        return j;
    const int p = 2 * n;
    int r = j % p;
    if (r < 0)
        r += p;
    return r >= n ? p - 1 - r : r;
}

/* Shared-memory column index with one padding word per 32: the phase-1
 * stores (V consecutive columns per thread) and the phase-2 reads (stride k)
 * then fall on distinct banks for V = 8, 16 and k = 2 .. 32 powers of two.
 * A group of V | 32 columns starting at a multiple of V shares one offset. */
__device__ __forceinline__ int skew(int c) { return c + (c >> 5); }

/* Packed two-lane fp32 operations (.f32x2, one issue slot for two lanes).
 * Each lane rounds once, as the scalar __fmul_rn / __fmaf_rn do.  Sums are
 * formed as fma(x, one, acc) with one = (1, 1) read from the launch
 * arguments, so the code generator cannot merge a product into them. */
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mov.b64 pc, {%6, %7};\n\t"
        "fma.rn.f32x2 pd, pa, pb, pc;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

/* Constants of the inexact-tap arithmetic, passed as launch arguments. */
struct PairConsts {
    float2 one;      // (1, 1)
    float2 m23;      // (-2^23, -2^23)
    float2 tap;      // (t, t)
    float2 ntap;     // (-t, -t)
};

/* Column accumulators of one thread: V adjacent input columns.
 * Exact taps (powers of two): sample sums only, as integers: for 8-bit
 * samples two 16-bit lanes per register (k * 255 < 2^16), columns (0, 2) and
 * (1, 3) of each 4-byte word; for 16-bit samples one register per column, or
 * two 16-bit lanes per word when k * (2^bitdepth - 1) < 2^16 (packed16).
 * Inexact taps: sample sums and product errors as fp32 pairs of adjacent
 * columns (both exact: integers below 2^24, and multiples of 2^-E below
 * 2^24 * 2^-E). */
template <typename T, bool kExactTap>
struct ColAcc {
    static constexpr int V = 16 / sizeof(T);
    unsigned s[8];
    float2 sx[V / 2];
    float2 ex[V / 2];

    __device__ __forceinline__ void reset()
    {
        if constexpr (kExactTap) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                s[i] = 0u;
        } else {
#pragma unroll
            for (int j = 0; j < V / 2; ++j) {
                sx[j] = make_float2(0.0f, 0.0f);
                ex[j] = make_float2(0.0f, 0.0f);
            }
        }
    }

    /* bits of 2^23 + sample v of the 16-byte vector, as fp32 */
    __device__ __forceinline__ static float magic(const uint4 &q, int v)
    {
        const unsigned w = v < V / 4 ? q.x : v < V / 2 ? q.y
                                   : v < 3 * V / 4 ? q.z : q.w;
        unsigned bits;
        if (sizeof(T) == 1)
            bits = __byte_perm(w, 0x4B000000u, 0x7540u | (unsigned)(v & 3));
        else
            bits = __byte_perm(w, 0x4B000000u, (v & 1) ? 0x7432u : 0x7410u);
        return __uint_as_float(bits);
    }

    __device__ __forceinline__ void add(const uint4 &q, bool packed16,
                                        const PairConsts &c)
    {
        if constexpr (kExactTap) {
            const unsigned w[4] = {q.x, q.y, q.z, q.w};
            if (sizeof(T) == 1) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[2 * j] += __byte_perm(w[j], 0u, 0x4240u);
                    s[2 * j + 1] += __byte_perm(w[j], 0u, 0x4341u);
                }
            } else if (packed16) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    s[j] += w[j];
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[2 * j] += w[j] & 0xffffu;
                    s[2 * j + 1] += w[j] >> 16;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < V / 2; ++j) {
                const float2 mb = make_float2(magic(q, 2 * j),
                                              magic(q, 2 * j + 1));
                const float2 x = fma2_rn(mb, c.one, c.m23);       // exact
                const float2 nprod = mul2_rn(x, c.ntap);          // -fl(x t)
                const float2 e = fma2_rn(x, c.tap, nprod);        // exact
                ex[j] = fma2_rn(e, c.one, ex[j]);
                sx[j] = fma2_rn(x, c.one, sx[j]);
            }
        }
    }

    /* sample sum of column v */
    __device__ __forceinline__ int col(int v, bool packed16) const
    {
        if constexpr (!kExactTap) {
            return __float2int_rn((v & 1) ? sx[v >> 1].y : sx[v >> 1].x);
        } else {
            if (sizeof(T) == 1) {
                const unsigned r = s[2 * (v >> 2) + (v & 1)];
                return (int)((v & 2) ? r >> 16 : r & 0xffffu);
            }
            if (packed16) {
                const unsigned r = s[v >> 1];
                return (int)((v & 1) ? r >> 16 : r & 0xffffu);
            }
            return (int)s[v];
        }
    }

    /* write the V column sums of group g to one output row's arrays */
    __device__ __forceinline__ void store(int *rowS, int *rowE, int g,
                                          bool packed16, float err_scale) const
    {
        const int base = skew(g * V);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            rowS[base + v] = col(v, packed16);
            if constexpr (!kExactTap) {
                const float e = (v & 1) ? ex[v >> 1].y : ex[v >> 1].x;
                rowE[base + v] = __float2int_rn(__fmul_rn(e, err_scale));
            }
        }
    }
};

/* V samples starting at column c0 of row rp, packed as a 16-byte vector
 * (little-endian, as a vector load would give); columns >= w read as 0. */
template <typename T, bool kVec>
__device__ __forceinline__ uint4 load_group(const T *rp, int c0, int w)
{
    if (kVec)
        return __ldg(reinterpret_cast<const uint4 *>(rp + c0));
    constexpr int V = 16 / sizeof(T);
    unsigned wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const unsigned x = (c0 + v < w) ? (unsigned)__ldg(rp + c0 + v) : 0u;
        wd[v * sizeof(T) / 4] |= x << (8 * ((v * sizeof(T)) & 3));
    }
    return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

/* K > 0: k fixed at compile time (2..8); K == 0: k = p.k at run time. */
template <typename T, int K, bool kExactTap, bool kVec>
__global__ void __launch_bounds__(kThreads)
ssim_decimate_kernel(const DecimateParams p)
{
    constexpr int V = 16 / sizeof(T);
    /* output rows whose K input rows fill one load batch (fixed k) */
    constexpr int kRowsPerBatch = K > 0 ? (kBatch / K > 0 ? kBatch / K : 1) : 1;
    extern __shared__ int shm[];
    int *sS = shm;                        // R rows of column sample sums
    int *sE = shm + p.R * p.pitch;        // R rows of column error sums

    const int plane = blockIdx.z & 1;
    const size_t f = blockIdx.z >> 1;
    /* select, not index: a run-time index into the parameter arrays would
     * copy them to local memory */
    const T *src = static_cast<const T *>(plane ? p.src[1] : p.src[0]) +
                   f * p.in_frame_elems;
    float *dst = (plane ? p.dst[1] : p.dst[0]) + f * p.out_frame_elems;
    const int k = K > 0 ? K : p.k;
    const int w = p.w, h = p.h, half = k >> 1;
    const int x0 = blockIdx.x * p.X;
    const int xn = min(p.X, p.sw - x0);
    const int y0 = blockIdx.y * p.R;
    const int rn = min(p.R, p.sh - y0);

    /* Input columns the tile's windows touch, after mirroring. */
    const int J0 = k * x0 - half;
    const int J1 = J0 + xn * k - 1;
    const bool interior = J0 >= 0 && J1 < w;
    int C0 = 0, C1 = w - 1;
    if (J0 >= -w && J1 < 2 * w) {
        C0 = max(J0, 0);
        C1 = min(J1, w - 1);
        if (J0 < 0)
            C1 = max(C1, min(w - 1, -1 - J0));
        if (J1 >= w)
            C0 = min(C0, max(0, 2 * w - 1 - J1));
    }
    const int Ca = kVec ? (C0 & ~(V - 1)) : C0;
    const int G = (C1 + 1 - Ca + V - 1) / V;

    const PairConsts pc = {p.one2, make_float2(-8388608.0f, -8388608.0f),
                           make_float2(p.tap, p.tap),
                           make_float2(-p.tap, -p.tap)};

    /* Phase 1: thread (g, sub) sums column group g over the k input rows of
     * output rows sub, sub + m, sub + 2m, ... */
    const int m = kThreads / G > 0 ? kThreads / G : 1;
    for (int t = threadIdx.x; t < G * m; t += kThreads) {
        const int g = t % G;
        const int sub = t / G;
        const int nr = sub < rn ? (rn - 1 - sub) / m + 1 : 0;
        const int c0 = Ca + g * V;
        const T *col0 = src + c0;
        ColAcc<T, kExactTap> acc;
        acc.reset();
        if (K > 0) {
            /* whole output rows per batch: kRowsPerBatch * K loads */
            for (int rb = 0; rb < nr; rb += kRowsPerBatch) {
                uint4 q[kRowsPerBatch][K > 0 ? K : 1];
#pragma unroll
                for (int b = 0; b < kRowsPerBatch; ++b) {
                    if (rb + b < nr) {
                        const int yb = k * (y0 + sub + (rb + b) * m) - half;
#pragma unroll
                        for (int i = 0; i < (K > 0 ? K : 1); ++i)
                            q[b][i] = load_group<T, kVec>(
                                col0 + (size_t)mirror2n(yb + i, h) * w,
                                0, w - c0);
                    }
                }
#pragma unroll
                for (int b = 0; b < kRowsPerBatch; ++b) {
                    if (rb + b < nr) {
#pragma unroll
                        for (int i = 0; i < (K > 0 ? K : 1); ++i)
                            acc.add(q[b][i], p.packed16, pc);
                        const int r = sub + (rb + b) * m;
                        acc.store(sS + r * p.pitch, sE + r * p.pitch, g,
                                  p.packed16, p.err_scale);
                        acc.reset();
                    }
                }
            }
        } else {
            /* run-time k: batches of kBatch input rows; input row u of this
             * thread is row i of its output row ri */
            const int total = nr * k;
            int ri0 = 0, i0 = 0;
            for (int u0 = 0; u0 < total; u0 += kBatch) {
                uint4 q[kBatch];
                int ri = ri0, i = i0;
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    if (u0 + j < total) {
                        const int y = k * (y0 + sub + ri * m) - half + i;
                        q[j] = load_group<T, kVec>(
                            col0 + (size_t)mirror2n(y, h) * w, 0, w - c0);
                    }
                    if (++i == k) {
                        i = 0;
                        ++ri;
                    }
                }
                ri = ri0;
                i = i0;
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const bool row_end = i == k - 1;
                    const int r = sub + ri * m;
                    if (++i == k) {
                        i = 0;
                        ++ri;
                    }
                    if (u0 + j < total) {
                        acc.add(q[j], p.packed16, pc);
                        if (row_end) {
                            acc.store(sS + r * p.pitch, sE + r * p.pitch, g,
                                      p.packed16, p.err_scale);
                            acc.reset();
                        }
                    }
                }
                ri0 = ri;
                i0 = i;
            }
        }
    }
    __syncthreads();

    /* Phase 2: each output adds its window's k columns and rounds once. */
    for (int r = 0; r < rn; ++r) {
        const int *rowS = sS + r * p.pitch;
        const int *rowE = sE + r * p.pitch;
        float *orow = dst + (size_t)(y0 + r) * p.sw;
        for (int xo = threadIdx.x; xo < xn; xo += kThreads) {
            const int x = x0 + xo;
            const int jb = k * x - half;
            int S = 0, E = 0;
            if (interior || (jb >= 0 && jb + k <= w)) {
                const int cb = jb - Ca;
                /* fixed k: the unrolled loop; run-time k: the second */
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    const int c = skew(cb + i);
                    S += rowS[c];
                    if (!kExactTap)
                        E += rowE[c];
                }
                for (int i = K; i < k; ++i) {
                    const int c = skew(cb + i);
                    S += rowS[c];
                    if (!kExactTap)
                        E += rowE[c];
                }
            } else {
                for (int i = 0; i < k; ++i) {
                    const int c = skew(mirror2n(jb + i, w) - Ca);
                    S += rowS[c];
                    if (!kExactTap)
                        E += rowE[c];
                }
            }
            float out;
            if (kExactTap)
                out = __fmul_rn(__int2float_rn(S), p.out_scale);
            else
                out = __fmul_rn(
                    __ll2float_rn(p.T * (long long)S - (long long)E),
                    p.out_scale);
            orow[x] = out;
        }
    }
}

/* 8-bit samples, k = 4 or 8, rows a multiple of 16 bytes: every window
 * either lies inside one 16-column group or straddles a group boundary with
 * k/2 columns on each side.  Each thread loads its group's 16 bytes from
 * each of the k input rows of an output row and forms the window partial
 * sums with dp4a (byte masks select the window's columns): the left half of
 * the straddling window, the inner windows, the right half of the next
 * straddling window.  The straddling window at the group's start adds the
 * left neighbour's right half, taken by shuffle from lane - 1; lane 0 (or the
 * first group of a block column) reloads that neighbour's last word, and
 * group 0 mirrors its own left half.  The last window of a row is always an
 * inner one (w even and a multiple of 16), so the right edge needs no
 * mirror.  Outputs are written as one 8-byte (k = 8) or 16-byte (k = 4)
 * store per thread.  No shared memory, no block barrier. */
template <int K>
__global__ void __launch_bounds__(kThreads)
ssim_decimate_u8_partials_kernel(const DecimateParams p)
{
    static_assert(K == 4 || K == 8, "window partials for k = 4 and 8");
    constexpr int kOut = 16 / K;          // windows starting in a group
    constexpr int kHalf = K / 2;
    const int plane = blockIdx.z & 1;
    const size_t f = blockIdx.z >> 1;
    const unsigned char *src =
        static_cast<const unsigned char *>(plane ? p.src[1] : p.src[0]) +
        f * p.in_frame_elems;
    float *dst = (plane ? p.dst[1] : p.dst[0]) + f * p.out_frame_elems;
    const int w = p.w, h = p.h;
    const int G = w >> 4;                 // groups per row
    const int Gb = p.X;                   // groups per block column
    const int m = kThreads / Gb;          // output rows walked side by side
    const int t = threadIdx.x;
    const int gi = t % Gb;
    const int sub = t / Gb;
    const int g = blockIdx.x * Gb + gi;
    const bool col_ok = sub < m && g < G;
    const int lane = t & 31;
    /* thread t - 1 holds group g - 1 of the same output row */
    const bool nb_in_warp = lane > 0 && gi > 0;
    const int y0 = blockIdx.y * p.R;
    const int rn = min(p.R, p.sh - y0);
    const int iters = (p.R + m - 1) / m;
    const unsigned char *colp = src + 16 * (size_t)g;

    for (int it = 0; it < iters; ++it) {
        const int r = sub + it * m;
        const bool act = col_ok && r < rn;
        const int yb = K * (y0 + r) - kHalf;
        uint4 q[K];
        unsigned prev[K];
        if (act) {
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const unsigned char *rp =
                    colp + (size_t)mirror2n(yb + i, h) * w;
                q[i] = __ldg(reinterpret_cast<const uint4 *>(rp));
                if (!nb_in_warp && g > 0)
                    prev[i] = __ldg(reinterpret_cast<const unsigned *>(rp) - 1);
            }
        }
        unsigned left = 0u, right = 0u, inner[kOut - 1];
#pragma unroll
        for (int j = 0; j < kOut - 1; ++j)
            inner[j] = 0u;
        if (act) {
#pragma unroll
            for (int i = 0; i < K; ++i) {
                if constexpr (K == 8) {
                    left = __dp4a(q[i].x, 0x01010101u, left);
                    inner[0] = __dp4a(q[i].y, 0x01010101u, inner[0]);
                    inner[0] = __dp4a(q[i].z, 0x01010101u, inner[0]);
                    right = __dp4a(q[i].w, 0x01010101u, right);
                } else {
                    left = __dp4a(q[i].x, 0x00000101u, left);
                    inner[0] = __dp4a(q[i].x, 0x01010000u, inner[0]);
                    inner[0] = __dp4a(q[i].y, 0x00000101u, inner[0]);
                    inner[1] = __dp4a(q[i].y, 0x01010000u, inner[1]);
                    inner[1] = __dp4a(q[i].z, 0x00000101u, inner[1]);
                    inner[2] = __dp4a(q[i].z, 0x01010000u, inner[2]);
                    inner[2] = __dp4a(q[i].w, 0x00000101u, inner[2]);
                    right = __dp4a(q[i].w, 0x01010000u, right);
                }
            }
        }
        const unsigned from_left = __shfl_up_sync(0xffffffffu, right, 1);
        if (act) {
            unsigned prev_right;
            if (nb_in_warp) {
                prev_right = from_left;
            } else if (g == 0) {
                prev_right = left;       // mirrored: [-k/2, 0) -> [0, k/2)
            } else {
                prev_right = 0u;
#pragma unroll
                for (int i = 0; i < K; ++i)
                    prev_right = __dp4a(prev[i], K == 8 ? 0x01010101u
                                                        : 0x01010000u,
                                        prev_right);
            }
            float o[kOut];
            o[0] = __fmul_rn(__uint2float_rn(prev_right + left), p.out_scale);
#pragma unroll
            for (int j = 1; j < kOut; ++j)
                o[j] = __fmul_rn(__uint2float_rn(inner[j - 1]), p.out_scale);
            float *orow = dst + (size_t)(y0 + r) * p.sw + kOut * g;
            if constexpr (K == 8)
                *reinterpret_cast<float2 *>(orow) = make_float2(o[0], o[1]);
            else
                *reinterpret_cast<float4 *>(orow) =
                    make_float4(o[0], o[1], o[2], o[3]);
        }
    }
}

/* Any k in 2..8, 8- or 16-bit samples, rows a multiple of 16 bytes: each
 * thread owns a chunk of 16k bytes (NS = WT * k samples, WT = 16 windows for
 * 8-bit samples, 8 for 16-bit) and loads it as k 16-byte vectors per input
 * row.  Chunk column c belongs to window (c + k/2) / k of the chunk: window 0
 * is the right half of a window that starts in the previous chunk, windows
 * 1..WT-1 lie inside, window WT is the left part of the next chunk's window
 * 0.  All window indices and byte masks are compile-time constants, so the
 * sample sums go straight into per-window registers with dp4a (bytes) or
 * dp2a (16-bit halves), and the product errors (inexact taps) into
 * per-window fp32 sums from packed fp32 pairs.  Window 0 adds the left
 * neighbour's window WT (shuffle from lane - 1); lane 0 of a warp and the
 * first chunk of a block column load the previous chunk's last vector with
 * their own rows, and chunk 0 mirrors its first k/2 columns.  The last
 * window of a row never leaves the row (w even), so the right edge needs no
 * mirror.
 *
 * Inexact taps end in fp32 alone: with Sw the window's sample sum (an
 * integer below 2^23) and Ew its exact error sum, s1 = fl(t * Sw) and its
 * error fma(Sw, t, -s1) are exact, so is d = error - Ew (both multiples of
 * 2^-E below 2^24 * 2^-E for k <= 7), and fl(s1 + d) is the one rounding of
 * t * Sw - Ew, as the int64 form of the header would give it.
 *
 * kStaged (k = 3, one block column spanning the row): the block's input rows
 * come into shared memory by bulk asynchronous copies on one mbarrier, and
 * the k vectors per row are read from there; a block whose copies did not
 * arrive within the time limit reads global memory instead.  Otherwise no
 * shared memory and no barrier. */
/* CTAs per SM the window kernel's register allocation must allow: 4
 * (64 registers) against 3 at 76-80 registers measured 4-9% faster at
 * k = 3 and 6, though some widths then spill a few bytes. */
#ifndef FSSIM_WIN_MINB
#define FSSIM_WIN_MINB 4
#endif
/* Shared-memory budget of the staged window kernel (k = 3): the block's
 * input rows and the mbarrier. */
constexpr size_t kStageMaxBytes = 48 * 1024;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}

/* The staged window kernel's tile: input row K*(y0 + r) - K/2 + i
 * (mirrored) of the plane at src goes to shared row r*K + i, r < rn, i < K,
 * one bulk copy per row issued by the lanes of warp 0, all completing on
 * one mbarrier placed after the K*R rows.  Every thread waits for the copies
 * for at most one second; returns true when all of them arrived in time in
 * every thread of the block (one vote). */
template <typename T, int K>
__device__ __forceinline__ bool stage_rows(const DecimateParams &p,
                                           const T *src, int y0, int rn,
                                           uint32_t tile)
{
    const uint32_t rowb = (uint32_t)p.w * (uint32_t)sizeof(T);
    const int nrows = K * rn;
    const uint32_t bar = tile + (uint32_t)(K * p.R) * rowb;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar)
                     : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0)
            asm volatile(
                "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                    bar),
                "r"((uint32_t)nrows * rowb + p.stage_extra_tx)
                : "memory");
        __syncwarp();
        for (int j = threadIdx.x; j < nrows; j += 32) {
            const int r = j / K, i = j - r * K;
            const T *row = src + (size_t)mirror2n(K * (y0 + r) - K / 2 + i,
                                                  p.h) * p.w;
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::"
                         "complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                             tile + (uint32_t)j * rowb),
                         "l"(reinterpret_cast<uint64_t>(row)), "r"(rowb),
                         "r"(bar)
                         : "memory");
        }
    }
    bool arrived = mbar_try_wait(bar, 0);
    if (!arrived) {
        const uint64_t t0 = global_ns();
        while (!(arrived = mbar_try_wait(bar, 0)) &&
               global_ns() - t0 < 1000000000ull) {
        }
    }
    return !__syncthreads_or(!arrived);
}

/* The window kernel's work for one block; kTile: the block's input rows
 * are in shared memory at tile (row r*K + i for output row r of the
 * block), else they are read from global memory. */
template <typename T, int K, bool kTile>
__device__ __forceinline__ void windows_rows(const DecimateParams &p,
                                             uint32_t tile)
{
    static_assert(K >= 2 && K <= 8, "window kernel for k = 2..8");
    constexpr bool kExact = (K & (K - 1)) == 0;
    constexpr int V = 16 / sizeof(T);     // samples per 16-byte vector
    constexpr int WT = V;                 // windows per chunk
    constexpr int NS = WT * K;            // samples per chunk
    constexpr int H = K / 2;
    constexpr int SPW = 4 / sizeof(T);    // samples per 32-bit word
    const int plane = blockIdx.z & 1;
    const size_t f = blockIdx.z >> 1;
    const T *src = static_cast<const T *>(plane ? p.src[1] : p.src[0]) +
                   f * p.in_frame_elems;
    float *dst = (plane ? p.dst[1] : p.dst[0]) + f * p.out_frame_elems;
    const int w = p.w, h = p.h;
    const int G = (p.sw + WT - 1) / WT;   // chunks per row
    const int Gb = p.X;                   // chunks per block column
    const int m = kThreads / Gb;
    const int t = threadIdx.x;
    const int gi = t % Gb;
    const int sub = t / Gb;
    const int g = blockIdx.x * Gb + gi;
    const bool col_ok = sub < m && g < G;
    const int lane = t & 31;
    const bool nb_in_warp = lane > 0 && gi > 0;
    const bool need_prev = !nb_in_warp && g > 0;
    const int y0 = blockIdx.y * p.R;
    const int rn = min(p.R, p.sh - y0);
    const int iters = (p.R + m - 1) / m;
    const T *chunk = src + (size_t)NS * g;
    /* vectors of this chunk inside the row (w is a multiple of V) */
    const int nvec = min(K, (w - NS * g) / V);
    const float2 one = p.one2;
    const float2 m23 = make_float2(-8388608.0f, -8388608.0f);
    const float2 tap2 = make_float2(p.tap, p.tap);
    const float2 ntap2 = make_float2(-p.tap, -p.tap);

    for (int it = 0; it < iters; ++it) {
        const int r = sub + it * m;
        const bool act = col_ok && r < rn;
        const int yb = K * (y0 + r) - H;
        unsigned S[WT + 1];
        float E[WT + 1];
#pragma unroll
        for (int i = 0; i <= WT; ++i) {
            S[i] = 0u;
            E[i] = 0.0f;
        }
        unsigned Sp = 0u;                 // previous chunk's window WT, or
        float Ep = 0.0f;                  // the mirror of this chunk's start
        if (act) {
            for (int i = 0; i < K; ++i) {
                uint4 q[K];
                uint4 qp = make_uint4(0u, 0u, 0u, 0u);
                if constexpr (kTile) {
                    const uint32_t ra =
                        tile + (uint32_t)((r * K + i) * w + NS * g) *
                                   (uint32_t)sizeof(T);
#pragma unroll
                    for (int v = 0; v < K; ++v)
                        q[v] = v < nvec ? lds128(ra + 16u * v)
                                        : make_uint4(0u, 0u, 0u, 0u);
                    if (need_prev)
                        qp = lds128(ra - 16u);
                } else {
                    const T *rp = chunk + (size_t)mirror2n(yb + i, h) * w;
#pragma unroll
                    for (int v = 0; v < K; ++v)
                        q[v] = v < nvec ? __ldg(reinterpret_cast<const uint4 *>(
                                              rp) + v)
                                        : make_uint4(0u, 0u, 0u, 0u);
                    if (need_prev)
                        qp = __ldg(reinterpret_cast<const uint4 *>(rp) - 1);
                }
#pragma unroll
                for (int v = 0; v < K; ++v) {
                    const unsigned wd[4] = {q[v].x, q[v].y, q[v].z, q[v].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int c0 = V * v + SPW * j;   // first sample
                        const int wa = (c0 + H) / K;
                        /* sample sums: the word's samples of window wa..wa+2 */
#pragma unroll
                        for (int dw = 0; dw < 3; ++dw) {
                            const int win = wa + dw;
                            /* dp4a: byte b of the mask weighs byte b of the
                             * word; dp2a_lo: bytes 0 and 1 of the mask weigh
                             * the word's two 16-bit halves */
                            unsigned msk = 0u;
#pragma unroll
                            for (int b = 0; b < SPW; ++b)
                                if ((c0 + b + H) / K == win)
                                    msk |= 1u << (8 * b);
                            if (win <= WT && msk != 0u) {
                                if constexpr (sizeof(T) == 1)
                                    S[win] = __dp4a(wd[j], msk, S[win]);
                                else
                                    S[win] = __dp2a_lo(wd[j], msk, S[win]);
                            }
                        }
                        if constexpr (!kExact) {
#pragma unroll
                            for (int pp = 0; pp < SPW / 2; ++pp) {
                                const int c = c0 + 2 * pp;
                                const float2 x = fma2_rn(
                                    make_float2(
                                        ColAcc<T, false>::magic(q[v], c - V * v),
                                        ColAcc<T, false>::magic(q[v],
                                                                c + 1 - V * v)),
                                    one, m23);
                                const float2 e = fma2_rn(
                                    x, tap2, mul2_rn(x, ntap2));
                                const int w0 = (c + H) / K;
                                const int w1 = (c + 1 + H) / K;
                                E[w0] = __fadd_rn(E[w0], e.x);
                                E[w1] = __fadd_rn(E[w1], e.y);
                            }
                        }
                    }
                }
                /* the samples outside this chunk that window 0 needs */
                if (need_prev || g == 0) {
                    const uint4 qs = need_prev ? qp : q[0];
#pragma unroll
                    for (int b = 0; b < H; ++b) {
                        const int c = need_prev ? V - H + b : b;
                        const unsigned wv = c < V / 4 ? qs.x
                                          : c < V / 2 ? qs.y
                                          : c < 3 * V / 4 ? qs.z : qs.w;
                        const unsigned sv =
                            sizeof(T) == 1 ? (wv >> (8 * (c & 3))) & 0xffu
                                           : (wv >> (16 * (c & 1))) & 0xffffu;
                        Sp += sv;
                        if constexpr (!kExact) {
                            const float xf = (float)sv;
                            const float pr = __fmul_rn(xf, p.tap);
                            Ep = __fadd_rn(Ep, __fmaf_rn(xf, p.tap, -pr));
                        }
                    }
                }
            }
        }
        const unsigned s_left = __shfl_up_sync(0xffffffffu, S[WT], 1);
        const float e_left = __shfl_up_sync(0xffffffffu, E[WT], 1);
        if (act) {
            if (nb_in_warp) {
                Sp = s_left;
                Ep = e_left;
            }
            float *orow = dst + (size_t)(y0 + r) * p.sw + WT * g;
            const int nout = min(WT, p.sw - WT * g);
            float o[WT];
#pragma unroll
            for (int i = 0; i < WT; ++i) {
                const unsigned Sw = i == 0 ? S[0] + Sp : S[i];
                if constexpr (kExact) {
                    o[i] = __fmul_rn(__uint2float_rn(Sw), p.out_scale);
                } else {
                    const float Ew = i == 0 ? __fadd_rn(E[0], Ep) : E[i];
                    /* the exact window sum t * Sw - Ew, Ew exact in fp32:
                     * s1 = fl(t * Sw), its error by FMA (exact), then
                     * d = error - Ew (exact) and one rounding of s1 + d */
                    const float sf = __fsub_rn(
                        __uint_as_float(Sw | 0x4b000000u), 8388608.0f);
                    const float s1 = __fmul_rn(sf, p.tap);
                    const float d =
                        __fsub_rn(__fmaf_rn(sf, p.tap, -s1), Ew);
                    o[i] = __fmul_rn(__fadd_rn(s1, d), p.inv_q);
                }
            }
            /* a thread's outputs are consecutive: whole chunks go out as
             * 16- or 8-byte stores where the row start allows it */
            const uintptr_t oa = reinterpret_cast<uintptr_t>(orow);
            if (nout == WT && oa % 16 == 0) {
#pragma unroll
                for (int i = 0; i < WT; i += 4)
                    *reinterpret_cast<float4 *>(orow + i) =
                        make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
            } else if (nout == WT && oa % 8 == 0) {
#pragma unroll
                for (int i = 0; i < WT; i += 2)
                    *reinterpret_cast<float2 *>(orow + i) =
                        make_float2(o[i], o[i + 1]);
            } else {
#pragma unroll
                for (int i = 0; i < WT; ++i)
                    if (i < nout)
                        orow[i] = o[i];
            }
        }
    }
}

/* The global-memory form of a staged block whose rows did not arrive in
 * time; kept out of line so that it costs the staged form no registers. */
template <typename T, int K>
__device__ __noinline__ void windows_rows_global(const DecimateParams p)
{
    windows_rows<T, K, false>(p, 0u);
}

template <typename T, int K, bool kStaged>
__global__ void __launch_bounds__(kThreads, FSSIM_WIN_MINB)
ssim_decimate_windows_kernel(const DecimateParams p)
{
    if constexpr (kStaged) {
        /* all input rows of the block in shared memory (p.R <= m, one row
         * of outputs per thread); if they did not arrive within the time
         * limit, the block reads global memory as the unstaged kernel does,
         * with the same results */
        extern __shared__ __align__(16) unsigned char stage_smem[];
        const uint32_t tile = smem_u32(stage_smem);
        const int plane = blockIdx.z & 1;
        const size_t f = blockIdx.z >> 1;
        const T *src = static_cast<const T *>(plane ? p.src[1] : p.src[0]) +
                       f * p.in_frame_elems;
        const int y0 = blockIdx.y * p.R;
        const int rn = min(p.R, p.sh - y0);
        if (stage_rows<T, K>(p, src, y0, rn, tile))
            windows_rows<T, K, true>(p, tile);
        else
            windows_rows_global<T, K>(p);
    } else {
        windows_rows<T, K, false>(p, 0u);
    }
}

/* Scale 1: the converted samples. */
template <typename T>
__global__ void __launch_bounds__(kThreads)
ssim_convert_kernel(const T *ref, const T *dist, float *ref_out,
                    float *dist_out, size_t n, float inv)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        ref_out[i] = __fmul_rn((float)ref[i], inv);
        dist_out[i] = __fmul_rn((float)dist[i], inv);
    }
}

template <typename T, int K, bool kExactTap, bool kVec>
cudaError_t launch(const DecimateParams &p, int n_frames, size_t smem,
                   cudaStream_t stream)
{
    auto kern = ssim_decimate_kernel<T, K, kExactTap, kVec>;
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    DecimateParams q = p;
    const size_t in_bytes = p.in_frame_elems * sizeof(T);
    for (int f0 = 0; f0 < n_frames; f0 += kMaxFramesPerLaunch) {
        const int nf = n_frames - f0 < kMaxFramesPerLaunch
                           ? n_frames - f0 : kMaxFramesPerLaunch;
        for (int s = 0; s < 2; ++s) {
            q.src[s] = static_cast<const unsigned char *>(p.src[s]) +
                       in_bytes * (size_t)f0;
            q.dst[s] = p.dst[s] + p.out_frame_elems * (size_t)f0;
        }
        const dim3 grid((p.sw + p.X - 1) / p.X, (p.sh + p.R - 1) / p.R,
                        2 * nf);
        kern<<<grid, kThreads, smem, stream>>>(q);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

/* Launch shape of the 8-bit window-partials kernel: p.X groups per block
 * column, p.R output rows per block. */
template <int K>
cudaError_t launch_partials(DecimateParams p, int n_frames,
                            cudaStream_t stream)
{
    const int G = p.w >> 4;
    p.X = G < kThreads ? G : kThreads;
    const int m = kThreads / p.X;
    p.R = 2 * m < p.sh ? 2 * m : p.sh;
    DecimateParams q = p;
    const size_t in_bytes = p.in_frame_elems;
    for (int f0 = 0; f0 < n_frames; f0 += kMaxFramesPerLaunch) {
        const int nf = n_frames - f0 < kMaxFramesPerLaunch
                           ? n_frames - f0 : kMaxFramesPerLaunch;
        for (int s = 0; s < 2; ++s) {
            q.src[s] = static_cast<const unsigned char *>(p.src[s]) +
                       in_bytes * (size_t)f0;
            q.dst[s] = p.dst[s] + p.out_frame_elems * (size_t)f0;
        }
        const dim3 grid((G + p.X - 1) / p.X, (p.sh + p.R - 1) / p.R, 2 * nf);
        ssim_decimate_u8_partials_kernel<K><<<grid, kThreads, 0, stream>>>(q);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

/* Launch shape of the window kernel: p.X chunks per block column, p.R output
 * rows per block. */
template <typename T, int K>
cudaError_t launch_windows(DecimateParams p, int n_frames, bool allow_stage,
                           cudaStream_t stream)
{
    constexpr int WT = 16 / sizeof(T);
    const int G = (p.sw + WT - 1) / WT;
    p.X = G < kThreads ? G : kThreads;
    const int m = kThreads / p.X;
    const size_t rowb = (size_t)p.w * sizeof(T);
    /* staged: k = 3, one block column spans the row, one row of outputs
     * per thread, the block's K*m input rows fit the shared-memory budget
     * (measured at k = 3 only: 720p and 4K 8-bit, 3-6% faster) */
    const bool staged = allow_stage && K == 3 && G <= kThreads &&
                        (size_t)K * m * rowb + 16 <= kStageMaxBytes;
    p.R = staged ? m : 2 * m;
    if (p.R > p.sh)
        p.R = p.sh;
    const size_t smem = staged ? (size_t)K * p.R * rowb + 16 : 0;
    DecimateParams q = p;
    const size_t in_bytes = p.in_frame_elems * sizeof(T);
    for (int f0 = 0; f0 < n_frames; f0 += kMaxFramesPerLaunch) {
        const int nf = n_frames - f0 < kMaxFramesPerLaunch
                           ? n_frames - f0 : kMaxFramesPerLaunch;
        for (int s = 0; s < 2; ++s) {
            q.src[s] = static_cast<const unsigned char *>(p.src[s]) +
                       in_bytes * (size_t)f0;
            q.dst[s] = p.dst[s] + p.out_frame_elems * (size_t)f0;
        }
        const dim3 grid((G + p.X - 1) / p.X, (p.sh + p.R - 1) / p.R, 2 * nf);
        bool launched = false;
        if constexpr (K == 3) {
            if (staged) {
                ssim_decimate_windows_kernel<T, K, true>
                    <<<grid, kThreads, smem, stream>>>(q);
                launched = true;
            }
        }
        if (!launched)
            ssim_decimate_windows_kernel<T, K, false>
                <<<grid, kThreads, 0, stream>>>(q);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

/* Which kernel takes a fixed scale on the vector path: the window kernel or
 * the general two-phase one (measured choice per sample type and scale;
 * FSSIM_KERNEL=general, =windows or =windows_direct in the environment
 * overrides it, the last one the window kernel without staging). */
enum class FixedPath { kAuto, kGeneral, kWindows, kWindowsDirect };
FixedPath fixed_path_override();

template <typename T, int K>
constexpr bool prefer_windows()
{
    /* measured at 4K: the general kernel's coalesced loads win for 8-bit
     * samples at k = 2 and 16-bit samples at k = 8 */
    return !(sizeof(T) == 1 && K == 2) && !(sizeof(T) == 2 && K == 8);
}

template <typename T, int K>
cudaError_t launch_fixed(const DecimateParams &p, bool vec, int n_frames,
                         size_t smem, cudaStream_t stream)
{
    constexpr bool kExact = (K & (K - 1)) == 0;
    if (vec) {
        const FixedPath o = fixed_path_override();
        const bool windows = o == FixedPath::kAuto ? prefer_windows<T, K>()
                                                   : o != FixedPath::kGeneral;
        if (windows)
            return launch_windows<T, K>(p, n_frames,
                                        o != FixedPath::kWindowsDirect,
                                        stream);
        return launch<T, K, kExact, true>(p, n_frames, smem, stream);
    }
    return launch<T, K, kExact, false>(p, n_frames, smem, stream);
}

/* All kernels for one sample type (defined in fssim_u8.cu / fssim_u16.cu). */
template <typename T>
cudaError_t dispatch(const DecimateParams &p, bool exact, bool vec,
                     int n_frames, size_t smem, cudaStream_t stream);

template <typename T>
cudaError_t dispatch_impl(const DecimateParams &p, bool exact, bool vec,
                          int n_frames, size_t smem, cudaStream_t stream)
{
    /* 8-bit, k = 4 or 8, 16-byte rows and 16-byte aligned outputs */
    if (sizeof(T) == 1 && vec && (p.k == 4 || p.k == 8) && p.w % 16 == 0 &&
        ((uintptr_t)p.dst[0] | (uintptr_t)p.dst[1]) % 16 == 0)
        return p.k == 4 ? launch_partials<4>(p, n_frames, stream)
                        : launch_partials<8>(p, n_frames, stream);
    switch (p.k) {
    case 2: return launch_fixed<T, 2>(p, vec, n_frames, smem, stream);
    case 3: return launch_fixed<T, 3>(p, vec, n_frames, smem, stream);
    case 4: return launch_fixed<T, 4>(p, vec, n_frames, smem, stream);
    case 5: return launch_fixed<T, 5>(p, vec, n_frames, smem, stream);
    case 6: return launch_fixed<T, 6>(p, vec, n_frames, smem, stream);
    case 7: return launch_fixed<T, 7>(p, vec, n_frames, smem, stream);
    case 8: return launch_fixed<T, 8>(p, vec, n_frames, smem, stream);
    default: break;
    }
    if (exact)
        return vec ? launch<T, 0, true, true>(p, n_frames, smem, stream)
                   : launch<T, 0, true, false>(p, n_frames, smem, stream);
    return vec ? launch<T, 0, false, true>(p, n_frames, smem, stream)
               : launch<T, 0, false, false>(p, n_frames, smem, stream);
}

template <typename T>
cudaError_t convert(const void *ref, const void *dist, float *ref_out,
                    float *dist_out, size_t n, float inv,
                    cudaStream_t stream);

} // namespace fssim

#endif /* FSSIM_KERNELS_CUH */
