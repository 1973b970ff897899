// Forward logsumexp, displacement and SVGD sweeps, their backward sweeps, merges and the top-k
// backward, double.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_FWD, double, 4, kLse)
TP_DP_LIST(TP_INST_FWD, double, 4, kDisp)
#define TP_INST_SVGD(DP, T) template void launch_fwd<T, DP, 4, kSvgd, false>(const SweepArgs&, cudaStream_t);
TP_DP_LIST(TP_INST_SVGD, double)
template void launch_fwd_merge<double, kLse>(const SweepArgs&, cudaStream_t);
template void launch_fwd_merge<double, kDisp>(const SweepArgs&, cudaStream_t);
template void launch_fwd_merge<double, kSvgd>(const SweepArgs&, cudaStream_t);
TP_DP_LIST(TP_INST_BWD, double, 4, kBLse, kRow, true, false)
TP_DP_LIST(TP_INST_BWD, double, 4, kBLse, kCol, true, false)
TP_DP_LIST(TP_INST_BWD, double, 4, kBDisp, kRow, true, false)
TP_DP_LIST(TP_INST_BWD, double, 4, kBDisp, kCol, true, false)
template void launch_bwd_merge<double, kBLse, kRow, true, false>(const SweepArgs&, cudaStream_t);
TP_DP_LIST(TP_INST_BWD, double, 4, kBLseSym, kRow, true, false)
template void launch_bwd_merge<double, kBLseSym, kRow, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBLse, kCol, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBDisp, kRow, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBDisp, kCol, true, false>(const SweepArgs&, cudaStream_t);
template void launch_topk_bwd<double>(const SweepArgs&, const SweepArgs&, const int64_t*, const void*, int*, int*,
                                     int*, int*, cudaStream_t);
}  // namespace tp
