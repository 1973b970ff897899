// Backward matmul replay sweeps, float: row sweep and column sweep(s) for every bucket.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_BWD_VALS, float, 4, kBMatmul)
TP_DP_LIST(TP_INST_BWD_VALS, float, 16, kBMatmul)
TP_DP_LIST(TP_INST_BWD_VALS, float, 64, kBMatmul)
template void launch_bwd_merge<float, kBMatmul, kRow, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<float, kBMatmul, kCol, true, true>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<float, kBMatmul, kCol, true, false>(const SweepArgs&, cudaStream_t);
template void launch_bwd_merge<float, kBMatmul, kCol, false, true>(const SweepArgs&, cudaStream_t);
}  // namespace tp
