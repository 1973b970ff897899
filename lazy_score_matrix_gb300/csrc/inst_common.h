// Macros that explicitly instantiate the launchers over the compiled buckets.
#pragma once

#include "tp_kernels.cuh"

#define TP_DP_LIST(X, ...) X(4, __VA_ARGS__) X(8, __VA_ARGS__) X(16, __VA_ARGS__) X(32, __VA_ARGS__) X(64, __VA_ARGS__)

// forward sweep, both AFFINE variants
#define TP_INST_FWD(DP, T, CP, MODE)                                                  \
    template void launch_fwd<T, DP, CP, MODE, false>(const SweepArgs&, cudaStream_t); \
    template void launch_fwd<T, DP, CP, MODE, true>(const SweepArgs&, cudaStream_t);

#define TP_INST_TOPK(DP, T, K)                                                  \
    template void launch_topk<T, DP, K, false>(const SweepArgs&, cudaStream_t); \
    template void launch_topk<T, DP, K, true>(const SweepArgs&, cudaStream_t);

#define TP_INST_BWD(DP, T, CP, MODE, SIDE, G, V) \
    template void launch_bwd<T, DP, CP, MODE, SIDE, G, V>(const SweepArgs&, cudaStream_t);

// matmul/softmax backward for one (DP, CP): the row sweep, and either the fused column sweep or
// its two halves, as chosen by fused_col_sweep().
#define TP_INST_BWD_VALS(DP, T, CP, MODE)                           \
    TP_INST_BWD(DP, T, CP, MODE, kRow, true, false)                 \
    TP_INST_BWD_VALS_COL_##DP##_##CP(DP, T, CP, MODE)

#define TP_COL_FUSED(DP, T, CP, MODE) TP_INST_BWD(DP, T, CP, MODE, kCol, true, true)
#define TP_COL_SPLIT(DP, T, CP, MODE) \
    TP_INST_BWD(DP, T, CP, MODE, kCol, true, false) TP_INST_BWD(DP, T, CP, MODE, kCol, false, true)
// fused_col_sweep(DP, CP) == (DP + CP <= 80)
#define TP_INST_BWD_VALS_COL_4_4 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_4_16 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_4_64 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_8_4 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_8_16 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_8_64 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_16_4 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_16_16 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_16_64 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_32_4 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_32_16 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_32_64 TP_COL_SPLIT
#define TP_INST_BWD_VALS_COL_64_4 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_64_16 TP_COL_FUSED
#define TP_INST_BWD_VALS_COL_64_64 TP_COL_SPLIT
