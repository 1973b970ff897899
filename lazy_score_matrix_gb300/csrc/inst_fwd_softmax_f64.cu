// Forward softmax sweeps, double: every padded feature width x value width x affine variant.
#include "inst_common.h"

namespace tp {
TP_DP_LIST(TP_INST_FWD, double, 4, kSoftmax)
TP_DP_LIST(TP_INST_FWD, double, 16, kSoftmax)
TP_DP_LIST(TP_INST_FWD, double, 64, kSoftmax)
template void launch_fwd_merge<double, kSoftmax>(const SweepArgs&, cudaStream_t);
}  // namespace tp
