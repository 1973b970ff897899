// Host-side launcher declarations. The definitions live with the kernels (tp_kernels.cuh) and are
// explicitly instantiated, bucket by bucket, in the inst_*.cu translation units, so the C-ABI
// translation unit compiles no kernel itself.
#pragma once

#include <cuda_runtime.h>

#include "tp_args.h"

namespace tp {

// Calls the user's launch hook (tp_set_launch_hook), if any, around every launch.
void launch_hook(const char* kernel, int phase, cudaStream_t s);
struct HookScope {
    const char* name;
    cudaStream_t s;
    HookScope(const char* n, cudaStream_t st) : name(n), s(st) { launch_hook(name, 0, s); }
    ~HookScope() { launch_hook(name, 1, s); }
};

// Launch with programmatic stream serialization: the kernel may start before the previous kernel on the
// stream has finished (its prologue overlaps that kernel's tail) and calls griddep_wait (tp_device.cuh) before
// it touches global memory. A launch error is left for cudaGetLastError, like a <<<>>> launch's.
template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <class T, int DP, int CP, int MODE, bool AFFINE>
void launch_fwd(const SweepArgs& a, cudaStream_t s);
template <class T, int MODE>
void launch_fwd_merge(const SweepArgs& a, cudaStream_t s);
template <class T, int DP, int K, bool AFFINE>
void launch_topk(const SweepArgs& a, cudaStream_t s);
template <class T, int K>
void launch_topk_merge(const SweepArgs& a, cudaStream_t s);
template <class T, int DP, int CP, int MODE, int SIDE, bool DO_G, bool DO_V>
void launch_bwd(const SweepArgs& a, cudaStream_t s);
template <class T, int MODE, int SIDE, bool DO_G, bool DO_V>
void launch_bwd_merge(const SweepArgs& a, cudaStream_t s);
template <class T>
void launch_topk_bwd(const SweepArgs& rows, const SweepArgs& cols, const int64_t* idx, const void* gv, int* count,
                     int* start, int* cursor, int* bucket, cudaStream_t s);

// Buckets compiled for: padded feature widths (4, 8, 16, 32, 64), value widths (4, 16, 64) and
// top-k list lengths (1, 4, 8, 16, 32).
constexpr int pad_bucket(int w) { return w <= 4 ? 4 : w <= 8 ? 8 : w <= 16 ? 16 : w <= 32 ? 32 : 64; }
constexpr int cpad_bucket(int w) { return w <= 4 ? 4 : w <= 16 ? 16 : 64; }
constexpr int kTopkMax = 32;
constexpr int topk_bucket(int k) { return k <= 1 ? 1 : k <= 4 ? 4 : k <= 8 ? 8 : k <= 16 ? 16 : 32; }
// Column sweeps of matmul/softmax compute dY and dV in one pass when the registers allow it.
constexpr bool fused_col_sweep(int DP, int CP) { return DP + CP <= 80; }

}  // namespace tp
