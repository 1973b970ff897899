// Forward matmul sweeps, float: every padded feature width x value width x affine variant.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_FWD, float, 4, kMatmul)
TP_DP_LIST(TP_INST_FWD, float, 16, kMatmul)
TP_DP_LIST(TP_INST_FWD, float, 64, kMatmul)
template void launch_fwd_merge<float, kMatmul>(const SweepArgs&, cudaStream_t);
}  // namespace tp
