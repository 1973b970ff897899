// Top-k sweeps and merges, float: every padded feature width x list length x affine variant.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_TOPK, float, 1)
TP_DP_LIST(TP_INST_TOPK, float, 4)
TP_DP_LIST(TP_INST_TOPK, float, 8)
TP_DP_LIST(TP_INST_TOPK, float, 16)
TP_DP_LIST(TP_INST_TOPK, float, 32)
template void launch_topk_merge<float, 1>(const SweepArgs&, cudaStream_t);
template void launch_topk_merge<float, 4>(const SweepArgs&, cudaStream_t);
template void launch_topk_merge<float, 8>(const SweepArgs&, cudaStream_t);
template void launch_topk_merge<float, 16>(const SweepArgs&, cudaStream_t);
template void launch_topk_merge<float, 32>(const SweepArgs&, cudaStream_t);
}  // namespace tp
