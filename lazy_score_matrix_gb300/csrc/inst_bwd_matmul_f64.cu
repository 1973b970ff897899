// Backward matmul replay sweeps, double: row sweep and column sweep(s) for every bucket.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_BWD_VALS, double, 4, kBMatmul)
TP_DP_LIST(TP_INST_BWD_VALS, double, 16, kBMatmul)
TP_DP_LIST(TP_INST_BWD_VALS, double, 64, kBMatmul)
template void launch_bwd_merge<double, kBMatmul, kRow, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBMatmul, kCol, true, true>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBMatmul, kCol, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<double, kBMatmul, kCol, false, true>(const SweepArgs&, cudaStream_t);
}  // namespace tp
