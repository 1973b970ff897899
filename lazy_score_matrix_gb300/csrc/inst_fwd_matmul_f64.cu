// Forward matmul sweeps, double: every padded feature width x value width x affine variant.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_FWD, double, 4, kMatmul)
TP_DP_LIST(TP_INST_FWD, double, 16, kMatmul)
TP_DP_LIST(TP_INST_FWD, double, 64, kMatmul)
template void launch_fwd_merge<double, kMatmul>(const SweepArgs&, cudaStream_t);
}  // namespace tp
