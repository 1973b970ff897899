// tp_pairwise_logsumexp_noalloc: the row log-sum-exp for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or have torch or another allocator do it) at the point where
// they need the result: code that runs inside another allocator's critical section or its
// out-of-memory callback, real-time loops that forbid any allocation after start-up, and hosts that
// embed this library without a way to size and own a workspace. This entry point needs no
// workspace argument. Its scratch (the per-split partial states of the streamed log-sum-exp) lives
// in a fixed array in device memory that belongs to this library: kNoAllocScratchBytes bytes, held
// on every GPU that loads the library until the process exits.
//
// Set-up: the first call on a device looks up the array's device address (cudaGetSymbolAddress, with
// that device current) and caches it; make that first call before any stream capture. Later calls
// on that device do no set-up.
//
// Sharing: every call on a device uses the same array, which keeps whatever the previous call left
// there. Nothing in it needs to start at zero: each call writes every partial state before reading
// it. Calls whose GPU work overlaps (different streams, or different host threads, without ordering
// between them) race on the array and give wrong results; order them on one stream or with events.
//
// The computation and every other convention are those of tp_pairwise_logsumexp, to which this entry
// point hands the array as its workspace.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "tp.h"

namespace tp {
void set_last_error(const std::string& msg);  // tp_api.cu: the text tp_last_error() returns
}

namespace {

// 16 MiB per device. The streamed (SIMT) log-sum-exp needs at most 2 MiB for any shape; the fp32 D = 64
// tensor-core path keeps an fp16 hi/lo copy of the points (256 bytes per point, once when Y is X) and
// 4 KiB of partials per row block of 128 rows plus 0.6 MiB, so it fits up to N = 54542 when Y is X and
// up to N + M of about 55000 when they differ. Larger problems are rejected by the size check below.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
tp_status scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        tp::set_last_error(std::string("no usable current CUDA device: ") + cudaGetErrorString(e));
        return TP_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            tp::set_last_error(std::string("cudaGetSymbolAddress of the scratch array failed: ") +
                               cudaGetErrorString(e));
            return TP_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return TP_OK;
}

}  // namespace

extern "C" {

TP_API tp_status tp_pairwise_logsumexp_noalloc(const tp_pairs* pairs, const tp_score* score, int exclude_self,
                                               void* lse, void* stream) {
    const size_t need = tp_workspace_size("pairwise_logsumexp", pairs, 0, 0);
    if (need == (size_t)-1) {
        tp::set_last_error("invalid sizes (the limits of tp_pairwise_logsumexp apply)");
        return TP_ERR_INVALID_ARG;
    }
    if (need > kNoAllocScratchBytes) {
        tp::set_last_error("problem needs " + std::to_string(need) + " bytes of scratch, above the " +
                           std::to_string(kNoAllocScratchBytes) +
                           "-byte fixed array of tp_pairwise_logsumexp_noalloc; call tp_pairwise_logsumexp with a "
                           "workspace instead");
        return TP_ERR_INVALID_ARG;
    }
    void* ws = nullptr;
    if (need > 0) {
        const tp_status s = scratch_for_current_device(&ws);
        if (s != TP_OK) return s;
    }
    return tp_pairwise_logsumexp(pairs, score, exclude_self, lse, ws, need > 0 ? kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"
