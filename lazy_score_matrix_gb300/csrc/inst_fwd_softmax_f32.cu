// Forward softmax sweeps, float: every padded feature width x value width x affine variant.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_FWD, float, 4, kSoftmax)
TP_DP_LIST(TP_INST_FWD, float, 16, kSoftmax)
TP_DP_LIST(TP_INST_FWD, float, 64, kSoftmax)
template void launch_fwd_merge<float, kSoftmax>(const SweepArgs&, cudaStream_t);
}  // namespace tp
