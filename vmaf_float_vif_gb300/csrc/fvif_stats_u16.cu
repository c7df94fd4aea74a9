/* Statistic kernels reading scale-0 U16 samples (ingest fused into the
 * loads).  Specialised tap counts: those of kernelscale 0.5, 1 and 2 at
 * scale 0; any other count takes the run-time-width variant. */
#include "fvif_dispatch.cuh"

namespace fvif {

cudaError_t stats_dispatch_u16(const StatsArgs &a, const Taps &tp,
                                cudaStream_t st)
{
    switch (tp.fixed_ok ? tp.n : 0) {
    case 9: return run_stats<9, SrcKind::U16>(a, tp, st);
    case 17: return run_stats<17, SrcKind::U16>(a, tp, st);
    case 35: return run_stats<35, SrcKind::U16>(a, tp, st);
    default: return run_stats<0, SrcKind::U16>(a, tp, st);
    }
}

} // namespace fvif
