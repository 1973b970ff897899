// Host-side helpers of the tensor-core kernels: TMA tensor-map encoding (through the driver entry
// point, so the library does not link libcuda) and workspace carving.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tp_launch.h"

namespace tp {

// The library's device error word on the current device (tp_status.cu), written by a bounded wait that
// gives up; nullptr (reason in tp_last_error) if its address cannot be looked up.
int* device_error_word();

namespace tc {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Row-major [rows, inner] fp32 with a 32-element (128-byte) box of box_rows rows, 128-byte swizzle;
// rows past the end read as zeros. inner * 4 must be a multiple of 16.
inline bool make_map_2d(CUtensorMap* m, const float* base, int64_t inner, int64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)inner * sizeof(float)};
    cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [rows, 64] point-major arrays
inline bool make_map_rows(CUtensorMap* m, const float* base, int64_t rows, int box_rows) {
    return make_map_2d(m, base, 64, rows, box_rows);
}
inline bool make_map(CUtensorMap* m, const float* base, int64_t rows) { return make_map_rows(m, base, rows, 128); }
// feature-major [64, cols] arrays (cols a multiple of 64): boxes of 32 columns x 64 feature rows
inline bool make_map_t(CUtensorMap* m, const float* base, int64_t cols) { return make_map_2d(m, base, cols, 64, 64); }

// Row-major [rows, 64] fp16 (128-byte rows) with boxes of the full row x box_rows rows, 128-byte swizzle;
// rows past the end read as zeros.
inline bool make_map_f16(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp16 hi/lo split of x 2^e per point row (the pre-pass of the kind::f16 kernels, tp_tc_lse.cu): hi and lo
// [rows][64] fp16, inv_scale = 2^-e and norm = |x|^2 for rows_pad rows (zeros past rows); cnt (optional):
// ncnt counters zeroed for the kernel that follows.
void launch_split16(const float* x, int64_t rows, int64_t rows_pad, void* hi, void* lo, float* inv_scale, float* norm,
                    int* cnt, int64_t ncnt, cudaStream_t s);

// The tile table pfx [RB + 1] of a masked schedule (tp_tc.cuh, Sched), built on the stream (tp_tc_lse.cu).
struct Sched;
void launch_sched_prefix(const Sched& sc, int64_t* pfx, cudaStream_t s);

inline size_t al256(size_t v) { return (v + 255) / 256 * 256; }

// Persistent grids: at most one CTA per SM of the current device (looked up once per device). Workspaces are
// sized for the GB300's 152 (shapes only); a device with fewer SMs runs that many CTAs over the same work.
inline int capped_grid(int g) {
    static int sms[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return g;
    if (!sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return g;
        sms[dev] = v;
    }
    return g < sms[dev] ? g : sms[dev];
}

}  // namespace tc
}  // namespace tp
