/* Statistic kernels reading the fp32 (ref, dist) planes of scales 1..3.
 * Specialised tap counts: those of kernelscale 0.5, 1 and 2 at scales 1..3;
 * any other count takes the run-time-width variant. */
#include "fvif_dispatch.cuh"

namespace fvif {

cudaError_t stats_dispatch_f2(const StatsArgs &a, const Taps &tp,
                              cudaStream_t st)
{
    switch (tp.fixed_ok ? tp.n : 0) {
    case 1: return run_stats<1, SrcKind::F2>(a, tp, st);
    case 3: return run_stats<3, SrcKind::F2>(a, tp, st);
    case 5: return run_stats<5, SrcKind::F2>(a, tp, st);
    case 7: return run_stats<7, SrcKind::F2>(a, tp, st);
    case 9: return run_stats<9, SrcKind::F2>(a, tp, st);
    case 11: return run_stats<11, SrcKind::F2>(a, tp, st);
    case 19: return run_stats<19, SrcKind::F2>(a, tp, st);
    default: return run_stats<0, SrcKind::F2>(a, tp, st);
    }
}

} // namespace fvif
