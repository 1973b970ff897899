// Backward softmax replay sweeps, double: row sweep and column sweep(s) for every bucket.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_BWD_VALS, double, 4, kBSoftmax)
TP_DP_LIST(TP_INST_BWD_VALS, double, 16, kBSoftmax)
TP_DP_LIST(TP_INST_BWD_VALS, double, 64, kBSoftmax)
template void launch_bwd_merge<double, kBSoftmax, kRow, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBSoftmax, kCol, true, true>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBSoftmax, kCol, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBSoftmax, kCol, false, true>(const SweepArgs&, cudaStream_t);
}  // namespace tp
