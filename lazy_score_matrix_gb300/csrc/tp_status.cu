// Device-side status of libtp: one error word per device that every bounded wait of the tensor-core
// kernels writes when it gives up, its read-back (tp_device_status), a self-test kernel whose bounded
// wait runs out on purpose (tp_selftest_bounded_wait), and host-side fault injection before launch.
//
// The tensor-core kernels are warp-specialised pipelines whose warps wait on one another through
// mbarriers. Every such wait is bounded (2 s): past the limit the waiting thread records a site code in
// the error word (the first code is kept), its warp leaves the tile loop, the CTA releases its tensor
// memory and the kernel returns. The results of that call are then wrong, and the caller learns of it
// only through tp_device_status after synchronising: the same status-and-check convention as the
// guide's solvers, which carry a status beside their result ("Using Torchpairwise in Models", What to
// Check). No kernel traps.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "tp.h"
#include "tp_device.cuh"
#include "tp_launch.h"
#include "tp_tc.cuh"

namespace tp {
void set_last_error(const std::string& msg);  // tp_api.cu
tp_status launched(int n);                    // tp_api.cu: counts launches, checks the launch error

namespace {

static __device__ __align__(256) int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int* g_word[kMaxDevices] = {};

// Site codes of the bounded waits (the second argument after the parity in each kernel's mbar_wait).
const char* site_text(int code) {
    if (code == tc::kSelfTestCode) return "the bounded-wait self-test (tp_selftest_bounded_wait)";
    if (code >= 11 && code <= 18) return "the tensor-core log-sum-exp forward (lse_fwd_tc)";
    if (code >= 21 && code <= 39) return "the tensor-core log-sum-exp backward (lse_bwd_sym_tc)";
    if (code >= 41 && code <= 59) return "a tensor-core attention sweep (attn_fwd_tc / attn_bwd_row_tc / attn_bwd_col_tc)";
    if (code >= 61 && code <= 79) return "the tensor-core log-sum-exp backward (lse_bwd_lin_tc)";
    if (code >= 81 && code <= 99) return "the tensor-core top-k (topk_tc)";
    return "a tensor-core kernel";
}

// One CTA of one warp: an mbarrier that expects one arrival and gets none, waited on with the given
// limit. Nothing else is in flight (no copy, no MMA, no tensor memory), so giving up is safe.
__global__ void bounded_wait_selftest(int* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::mbar_fence_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, err, tc::kSelfTestCode, limit_ns);
}

// y = the fp64 exp the kernels use (exp_table), element by element.
__global__ void exp64_selftest(const double* __restrict__ x, double* __restrict__ y, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = ExpTraits<double>::exp(x[i]);
}

}  // namespace

// Device address of the error word on the current device (looked up once per device), or nullptr with
// the reason in tp_last_error().
int* device_error_word() {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_last_error(std::string("no usable current CUDA device: ") + cudaGetErrorString(e));
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_word[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_error);
        if (e != cudaSuccess || !p) {
            set_last_error(std::string("cudaGetSymbolAddress of the device error word failed: ") +
                           cudaGetErrorString(e));
            return nullptr;
        }
        g_word[dev] = static_cast<int*>(p);
    }
    return g_word[dev];
}

// TP_FAULT_INJECT=<entry> (the entry point's name without "tp_", e.g. "pairwise_logsumexp") makes that
// entry fail with TP_ERR_CUDA after validating its arguments and before launching anything, as if the
// launch had failed. Read on every call, so a test can set and clear it while the process runs.
tp_status injected_fault(const char* entry) {
    const char* v = getenv("TP_FAULT_INJECT");
    if (!v || !*v || std::strcmp(v, entry) != 0) return TP_OK;
    set_last_error(std::string("fault injected before launch (TP_FAULT_INJECT=") + v + ")");
    return TP_ERR_CUDA;
}

}  // namespace tp

extern "C" {

TP_API tp_status tp_device_status(int reset) {
    int* w = tp::device_error_word();
    if (!w) return TP_ERR_CUDA;
    int code = 0;
    cudaError_t e = cudaMemcpy(&code, w, sizeof code, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && reset && code != 0) {
        const int zero = 0;
        e = cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
        tp::set_last_error(std::string("tp_device_status: ") + cudaGetErrorString(e));
        return TP_ERR_CUDA;
    }
    if (code == 0) return TP_OK;
    tp::set_last_error("a bounded wait in " + std::string(tp::site_text(code)) + " gave up (site code " +
                       std::to_string(code) + "); the results of that call are invalid");
    return TP_ERR_TIMEOUT;
}

TP_API tp_status tp_selftest_bounded_wait(int64_t limit_ns, void* stream) {
    if (limit_ns < 1000 || limit_ns > (int64_t)tp::tc::kWaitNs) {
        tp::set_last_error("tp_selftest_bounded_wait: limit_ns must be in [1000, 2e9]");
        return TP_ERR_INVALID_ARG;
    }
    int* w = tp::device_error_word();
    if (!w) return TP_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        tp::HookScope h("bounded_wait_selftest", s);
        tp::bounded_wait_selftest<<<1, 32, 0, s>>>(w, (unsigned long long)limit_ns);
    }
    return tp::launched(1);
}

TP_API tp_status tp_selftest_exp64(const double* x, double* y, int64_t n, void* stream) {
    if (n < 0 || (n > 0 && (!x || !y))) {
        tp::set_last_error("tp_selftest_exp64: x and y must be device arrays of n >= 0 doubles");
        return TP_ERR_INVALID_ARG;
    }
    if (n == 0) return TP_OK;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        tp::HookScope h("exp64_selftest", s);
        tp::exp64_selftest<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, y, n);
    }
    return tp::launched(1);
}

}  // extern "C"
