/*
 * fvif_dec_tma.cuh -- the first decimation (integer samples -> scale 1)
 * with its source tile staged in shared memory by the Tensor Memory
 * Accelerator.
 *
 * Same outputs, bit for bit, as decimate_kernel<N, U8|U16>: the vertical
 * filter with the taps of scale 1 at the even source rows, then the
 * horizontal filter at the even columns, reflect-then-clamp boundary
 * ("ADR-1444 ...", Context and Decision), every product and sum rounded
 * once in the same order.  Only the way the samples reach the arithmetic
 * differs: instead of one 1- or 2-byte global load per sample and thread,
 * one thread issues two 3-D tensor copies (ref and dist planes) of the
 * CTA's whole source tile into shared memory, completing on an mbarrier,
 * and the vertical pass reads the tile from there.
 *
 * Tile geometry (per CTA: kDY decimated rows, dec_cols(R) decimated
 * columns, as decimate_kernel):
 *  - source rows ys = 2*y0 - R .. ys + BH - 1, BH = 2*kDY + 2R - 1;
 *  - source columns xs .. xs + BW - 1, where xs = 2*x0 - R rounded down to
 *    a multiple of 16 bytes of samples (a tensor copy must start on a
 *    16-byte boundary in x), BW = the tile's 127 columns plus that
 *    rounding, rounded up to 16 bytes.
 * Coordinates outside the plane (the first and last tiles) are filled with
 * zeros by the copy; every sample an output needs comes from a reflected
 * index, which lies inside the tile whenever the plane is at least 2R + 2
 * samples wide and high (the host checks this), and every shared-memory
 * index is clamped into the tile as well.
 *
 * Waits are bounded: a thread that has not seen the tile arrive after one
 * second (global timer) gives up; the CTA agrees on that with one vote,
 * sets bit 0 of *status and returns without touching its outputs.  No
 * thread ever spins without a limit.
 */
#pragma once

#include <cuda.h>

#include <type_traits>

#include "fvif_kernels.cuh"

namespace fvif {

/* Tile width in samples for element size EB and half-width R. */
__host__ __device__ constexpr int dtma_align(int eb) { return 16 / eb; }
__host__ __device__ constexpr int dtma_bw(int r, int eb)
{
    return (dec_width(r) + dtma_align(eb) - 1 + dtma_align(eb) - 1) /
           dtma_align(eb) * dtma_align(eb);
}
__host__ __device__ constexpr int dtma_bh(int r) { return 2 * kDY + 2 * r - 1; }
__host__ __device__ constexpr size_t dtma_tile_bytes(int r, int eb)
{
    return (size_t)dtma_bw(r, eb) * dtma_bh(r) * eb;
}
/* dynamic shared memory: the two sample tiles (128-byte aligned), reused
 * for the vertically filtered rows Vd once the tiles have been read, then
 * the local row table */
/* float2 per row of the vertically filtered tile Vd: its 127 columns and
 * what the horizontal items read, a multiple of 2 so that every item's
 * first column is 16-byte aligned */
constexpr int kVdPitch = 130;
__host__ __device__ constexpr int dtma_vd_pitch(int) { return kVdPitch; }
/* Placement of the filtered columns in a Vd row for the two-output
 * horizontal items (up to 9 taps): 16-byte pair p of a row is stored at
 * pair p ^ bit3(p), so the eight pairs a quarter warp reads in one load
 * (every second pair of a run of sixteen) fall on distinct bank groups;
 * column c (a float2) moves with its pair.  Wider kernels keep the plain
 * layout. */
template <int N>
__device__ __forceinline__ int dtma_swz_pair(int p)
{
    return N <= 9 ? p ^ ((p >> 3) & 1) : p;
}
template <int N>
__device__ __forceinline__ int dtma_swz(int c)
{
    return N <= 9 ? c ^ (((c >> 4) & 1) << 1) : c;
}

__host__ __device__ constexpr size_t dtma_main_bytes(int r, int eb)
{
    return 2 * ((dtma_tile_bytes(r, eb) + 127) / 128 * 128) >
                   sizeof(float2) * kDY * (size_t)dtma_vd_pitch(r)
               ? 2 * ((dtma_tile_bytes(r, eb) + 127) / 128 * 128)
               : sizeof(float2) * kDY * (size_t)dtma_vd_pitch(r);
}
__host__ __device__ constexpr size_t dtma_rows_offset(int r, int eb)
{
    return dtma_main_bytes(r, eb);
}
/* the mbarrier, 8-byte aligned, after the row table */
__host__ __device__ constexpr size_t dtma_bar_offset(int r, int eb)
{
    return (dtma_rows_offset(r, eb) + sizeof(int) * (2 * kDY + 2 * r) + 7) /
           8 * 8;
}
__host__ __device__ constexpr size_t dtma_smem_bytes(int r, int eb)
{
    return dtma_bar_offset(r, eb) + sizeof(uint64_t);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

/* Vertical pass of one item from the shared-memory tiles: kDRV outputs at
 * local rows 2i of the item.  Row t of the item is at element idx + t*BW
 * (kInRows) or at rl[t] + idx. */
template <int N, SrcKind K, bool kInRows, typename T>
__device__ __forceinline__ void dtma_vitem(const T *tx, const T *ty,
                                           const int *rl, int idx, int BW,
                                           const Taps &tp,
                                           float2 (&acc)[kDRV])
{
    constexpr bool kRaw = K == SrcKind::U16;
#pragma unroll
    for (int t = 0; t < 2 * (kDRV - 1) + N; ++t) {
        const int e = kInRows ? idx : rl[t] + idx;
        if constexpr (kInRows)
            idx += BW;
        const float2 v = make_float2(__uint2float_rn(tx[e]),
                                     __uint2float_rn(ty[e]));
#pragma unroll
        for (int i = 0; i < kDRV; ++i) {
            const int k = t - 2 * i;
            if (k >= 0 && k < N) {
                const int kk = fold(k, N);
                const float2 p = mul2_rn(kRaw ? tp.ra2[kk] : tp.t2[kk], v);
                acc[i] = (k == 0) ? p : acc2_rn(acc[i], p, tp.one2);
            }
        }
    }
}

template <int N, SrcKind K>
__global__ void __launch_bounds__(kDecThreads)
    decimate_tma_kernel(const __grid_constant__ CUtensorMap tmx,
                        const __grid_constant__ CUtensorMap tmy,
                        const DecArgs a, const Taps tp)
{
    using T = typename std::conditional<K == SrcKind::U8, uint8_t,
                                        uint16_t>::type;
    constexpr int EB = sizeof(T);
    constexpr int R = N / 2;
    constexpr int DX = dec_cols(R);
    constexpr int DW = dec_width(R);
    constexpr int BW = dtma_bw(R, EB);
    constexpr int BH = dtma_bh(R);
    constexpr int VP = dtma_vd_pitch(R);
    constexpr uint32_t kTileBytes = (uint32_t)dtma_tile_bytes(R, EB);
    constexpr size_t kTileStride = (dtma_tile_bytes(R, EB) + 127) / 128 * 128;
    static_assert(N > 0 && N <= kMaxFixedTaps, "fixed widths only");
    static_assert((BW * EB) % 16 == 0 && BW <= 256 && BH <= 256,
                  "tensor-copy box");

    /* dynamic shared memory only (its base is 16-byte aligned, as a
     * tensor copy without swizzling needs): tiles | row table | mbarrier */
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T *tx = reinterpret_cast<T *>(smem_raw);
    T *ty = reinterpret_cast<T *>(smem_raw + kTileStride);
    float2 *Vd = reinterpret_cast<float2 *>(smem_raw);
    int *rl = reinterpret_cast<int *>(smem_raw + dtma_rows_offset(R, EB));
    uint64_t &bar =
        *reinterpret_cast<uint64_t *>(smem_raw + dtma_bar_offset(R, EB));

    const int W = a.w, H = a.h, W2 = W / 2, H2 = H / 2;
    const int x0 = blockIdx.x * DX, y0 = blockIdx.y * kDY, f = blockIdx.z;
    const int p0 = 2 * x0 - R;
    const int xs = p0 & ~(dtma_align(EB) - 1); /* floor, also below 0 */
    const int ys = 2 * y0 - R;

    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                         smem_addr(&bar))
                     : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        asm volatile(
            "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                smem_addr(&bar)),
            "r"(2 * kTileBytes + a.extra_tx)
            : "memory");
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile"
                     ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}],"
                     " [%5];" ::"r"(smem_addr(tx)),
                     "l"(reinterpret_cast<uint64_t>(&tmx)), "r"(xs), "r"(ys),
                     "r"(f), "r"(smem_addr(&bar))
                     : "memory");
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile"
                     ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}],"
                     " [%5];" ::"r"(smem_addr(ty)),
                     "l"(reinterpret_cast<uint64_t>(&tmy)), "r"(xs), "r"(ys),
                     "r"(f), "r"(smem_addr(&bar))
                     : "memory");
    }
    /* local row of source row ys + t (reflected, clamped into the tile) */
    for (int t = threadIdx.x; t < 2 * kDY + 2 * R - 1; t += kDecThreads)
        rl[t] = min(max(bound_index(ys + t, H) - ys, 0), BH - 1) * BW;

    /* wait for both tiles, for at most one second */
    bool arrived = mbar_try_wait(&bar, 0);
    if (!arrived) {
        const uint64_t t0 = global_ns();
        while (!(arrived = mbar_try_wait(&bar, 0)) &&
               global_ns() - t0 < 1000000000ull) {
        }
    }
    /* every thread also passes this barrier after the row table is made */
    if (__syncthreads_or(!arrived)) {
        if (threadIdx.x == 0 && a.status)
            atomicOr(a.status, 1u);
        return;
    }

    /* rows ys .. ys + BH - 1 all inside the plane: no reflection */
    const bool rows_in = ys >= 0 && ys + BH <= H;
    constexpr int NG = kDY / kDRV;
    static_assert(DW * NG <= kDecThreads, "one vertical item per thread");
    const int item = threadIdx.x;
    float2 acc[kDRV];
    const bool has_item = item < DW * NG;
    if (has_item) {
        const int cl = item % DW;
        const int g = item / DW;
        const int lc = min(max(bound_index(p0 + cl, W) - xs, 0), BW - 1);
        if (rows_in)
            dtma_vitem<N, K, true>(tx, ty, nullptr, (2 * g * kDRV) * BW + lc,
                                   BW, tp, acc);
        else
            dtma_vitem<N, K, false>(tx, ty, rl + 2 * g * kDRV, lc, BW, tp,
                                    acc);
    }
    __syncthreads(); /* the tiles are read; Vd reuses their memory */
    if (has_item) {
        const int cl = item % DW;
        const int g = item / DW;
#pragma unroll
        for (int i = 0; i < kDRV; ++i)
            Vd[(g * kDRV + i) * VP + dtma_swz<N>(cl)] = acc[i];
    }
    __syncthreads();
    float2 *dst = a.dst + (size_t)f * a.dst_frame_elems;
    if constexpr (N > 9) {
        /* wide kernels: one output per item (two would hold 2N+4 registers
         * of columns and cost occupancy) */
        for (int it = threadIdx.x; it < kDY * DX; it += kDecThreads) {
            const int yl = it / DX, xl = it % DX;
            const int yd = y0 + yl, xd = x0 + xl;
            if (yd >= H2 || xd >= W2)
                continue;
            const float2 *in = Vd + yl * VP + 2 * xl;
            float2 sum;
#pragma unroll
            for (int k = 0; k < N; ++k) {
                const float2 p = mul2_rn(tp.t2[k], in[k]);
                sum = (k == 0) ? p : acc2_rn(sum, p, tp.one2);
            }
            dst[(size_t)yd * W2 + xd] = sum;
        }
        return;
    }
    /* horizontal pass: two adjacent outputs per item, their N + 2 filtered
     * columns read as 16-byte pairs of float2; items run along a row */
    constexpr int kHI = (DX + 1) / 2;       /* two-output items per row */
    constexpr int kPairs = (N + 3) / 2;     /* 16-byte reads per item   */
    static_assert(2 * 2 * (kHI - 1) + 2 * kPairs <= kVdPitch,
                  "Vd reads stay inside a row");
    for (int it = threadIdx.x; it < kDY * kHI; it += kDecThreads) {
        const int yl = it / kHI, xl = (it - yl * kHI) * 2;
        const int yd = y0 + yl;
        if (yd >= H2)
            continue;
        const float4 *row = reinterpret_cast<const float4 *>(Vd + yl * VP);
        float2 col[2 * kPairs];
#pragma unroll
        for (int u = 0; u < kPairs; ++u) {
            const float4 v = row[dtma_swz_pair<N>(xl + u)];
            col[2 * u] = make_float2(v.x, v.y);
            col[2 * u + 1] = make_float2(v.z, v.w);
        }
        /* both outputs inside the row and a 16-byte aligned pair (even
         * row length, aligned plane): one vector store */
        if (DX % 2 == 0 && (W2 & 1) == 0 && x0 + xl + 1 < W2 &&
            (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
            float2 sum[2];
#pragma unroll
            for (int o = 0; o < 2; ++o) {
#pragma unroll
                for (int k = 0; k < N; ++k) {
                    const float2 p = mul2_rn(tp.t2[k], col[2 * o + k]);
                    sum[o] = (k == 0) ? p : acc2_rn(sum[o], p, tp.one2);
                }
            }
            *reinterpret_cast<float4 *>(dst + (size_t)yd * W2 + x0 + xl) =
                make_float4(sum[0].x, sum[0].y, sum[1].x, sum[1].y);
            continue;
        }
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            const int xd = x0 + xl + o;
            if (xl + o >= DX || xd >= W2)
                break;
            float2 sum;
#pragma unroll
            for (int k = 0; k < N; ++k) {
                const float2 p = mul2_rn(tp.t2[k], col[2 * o + k]);
                sum = (k == 0) ? p : acc2_rn(sum, p, tp.one2);
            }
            dst[(size_t)yd * W2 + xd] = sum;
        }
    }
}

} // namespace fvif

