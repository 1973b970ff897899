// Backward softmax replay sweeps, float: row sweep and column sweep(s) for every bucket.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_BWD_VALS, float, 4, kBSoftmax)
TP_DP_LIST(TP_INST_BWD_VALS, float, 16, kBSoftmax)
TP_DP_LIST(TP_INST_BWD_VALS, float, 64, kBSoftmax)
template void launch_bwd_merge<float, kBSoftmax, kRow, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<float, kBSoftmax, kCol, true, true>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<float, kBSoftmax, kCol, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<float, kBSoftmax, kCol, false, true>(const SweepArgs&, cudaStream_t);
}  // namespace tp
