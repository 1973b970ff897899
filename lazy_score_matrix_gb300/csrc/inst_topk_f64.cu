// Top-k sweeps and merges, double: every padded feature width x list length x affine variant.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_TOPK, double, 1)
TP_DP_LIST(TP_INST_TOPK, double, 4)
TP_DP_LIST(TP_INST_TOPK, double, 8)
TP_DP_LIST(TP_INST_TOPK, double, 16)
TP_DP_LIST(TP_INST_TOPK, double, 32)
template void launch_topk_merge<double, 1>(const SweepArgs&, cudaStream_t);
template void launch_topk_merge<double, 4>(const SweepArgs&, cudaStream_t);
template void launch_topk_merge<double, 8>(const SweepArgs&, cudaStream_t);
template void launch_topk_merge<double, 16>(const SweepArgs&, cudaStream_t);
template void launch_topk_merge<double, 32>(const SweepArgs&, cudaStream_t);
}  // namespace tp
