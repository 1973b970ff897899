// Measured arithmetic peaks of the current GPU, for the roofline denominators of the streamed (SIMT)
// kernels: fp32 FMA, fp64 FMA and the hardware base-2 exponential (the special-function unit), each
// timed with CUDA events around one kernel that keeps every SM busy with independent chains of
// dependent operations. Not part of libtp's C ABI: a calibration library the benchmark loads.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kChains = 8;  // independent dependency chains per thread (enough to cover the pipe latency)

template <class T>
__global__ void __launch_bounds__(256) fma_chains(T* sink, int64_t iters, T b, T c) {
    T a[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) a[k] = (T)(threadIdx.x + k) * (T)1e-3;
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kChains; ++k) a[k] = fma(a[k], b, c);
    }
    T s = 0;
#pragma unroll
    for (int k = 0; k < kChains; ++k) s += a[k];
    if (s == (T)-12345.678) sink[blockIdx.x] = s;  // never true for these inputs; keeps the work alive
}

__global__ void __launch_bounds__(256) ex2_chains(float* sink, int64_t iters) {
    float a[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) a[k] = -1e-3f * (float)(threadIdx.x + k);
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kChains; ++k) {
            float y;
            asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(a[k]));
            a[k] = -y;  // stays in [-1, 0): 2^a in [0.5, 1)
        }
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kChains; ++k) s += a[k];
    if (s == -12345.678f) sink[blockIdx.x] = s;
}

}  // namespace

extern "C" {

// kind 0: fp32 FMA, 1: fp64 FMA (TFLOP/s, 2 flop per FMA); 2: ex2.approx (Tera-ops/s). Runs `blocks_per_sm`
// blocks of 256 threads per SM for `iters` iterations of kChains operations per thread, after one warm-up
// launch. Returns the rate of the timed launch, or a negative value on a CUDA error. *ms receives its
// duration.
__attribute__((visibility("default"))) double tpk_peak(int kind, int64_t iters, int blocks_per_sm, float* ms) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1.0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1.0;
    const int grid = sms * blocks_per_sm;
    void* sink = nullptr;
    if (cudaMalloc(&sink, (size_t)grid * 8) != cudaSuccess) return -1.0;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    float t = 0.f;
    for (int rep = 0; rep < 2; ++rep) {  // the first launch warms up (clocks, instruction cache)
        cudaEventRecord(e0);
        if (kind == 0) fma_chains<float><<<grid, 256>>>(static_cast<float*>(sink), iters, 0.999f, 1e-4f);
        else if (kind == 1) fma_chains<double><<<grid, 256>>>(static_cast<double*>(sink), iters, 0.999, 1e-4);
        else ex2_chains<<<grid, 256>>>(static_cast<float*>(sink), iters);
        cudaEventRecord(e1);
        cudaEventSynchronize(e1);
        cudaEventElapsedTime(&t, e0, e1);
    }
    const cudaError_t err = cudaGetLastError();
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(sink);
    if (err != cudaSuccess || t <= 0.f) return -1.0;
    if (ms) *ms = t;
    const double ops = (double)grid * 256.0 * (double)iters * kChains * (kind == 2 ? 1.0 : 2.0);
    return ops / (t * 1e-3) / 1e12;
}

}  // extern "C"
