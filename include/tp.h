/*
 * libtp: streamed pairwise score consumers for GB300 (sm_103a).
 *
 * A pairwise score S[i,j] = f(x_i, y_j) over X [N,D] and Y [M,D] is evaluated tile by tile on the
 * GPU and consumed in the same pass; the [N,M] matrix is never stored. First derivatives re-evaluate
 * the pairs ("replay") in a row sweep (dX, row parameters) and a transposed column sweep (dY, dV,
 * column parameters), without atomics. Source of the method: "Using Torchpairwise in Models"
 * (torchpairwise guide, ml.html), introduction: bind scores lazily, consume them in bounded tiles or
 * fused CUDA kernels, never store the matrix, replay tiles for first derivatives; memory scales with
 * (N+M)*(D+C) plus a tile workspace.
 *
 * Canonical score (the guide's "Score Expressions" section: scalar scale, add_rows, add_columns,
 * weight_rows, weight_columns and exp are the fused nodes; this library fixes their order):
 *     base_ij = |x_i - y_j|^2                  (TP_SQEUCLIDEAN)
 *             | x_i . y_j                      (TP_LINEAR)
 *             | exp(-gamma |x_i - y_j|^2)      (TP_RBF; "Stein Variational Gradient Descent")
 *     t_ij    = scale * wr_i * wc_j * base_ij + br_i + bc_j   (absent weight = 1, absent bias = 0)
 *     S_ij    = apply_exp ? exp(t_ij) : t_ij
 *
 * Conventions shared by every entry point
 *   - Layout: every matrix is row-major and contiguous. X [N,D], Y [M,D], V [M,C], outputs [N,*],
 *     column gradients [M,*]. All element pointers have the dtype of `tp_pairs.dtype` (float or
 *     double) except top-k indices, which are int64.
 *   - Sizes: N, M >= 1; 1 <= D <= 64; 1 <= C <= 64 (the guide's fused range, "Task Map"); M and N
 *     below 2^31.
 *   - Memory: every pointer is caller-owned DEVICE memory (tp_pairs, tp_score and the scalar
 *     arguments themselves are host structs read during the call). libtp allocates nothing,
 *     frees nothing and never synchronises: all work is enqueued on `stream` (a cudaStream_t passed
 *     as void*, NULL = legacy default stream) and the call returns as soon as it is enqueued.
 *   - Workspace: `ws` is caller-owned device scratch of at least tp_workspace_size(entry, ...) bytes,
 *     aligned to 256 bytes (what cudaMalloc returns). Its size depends on the shapes only. It may be
 *     NULL when the required size is 0. The contents need no initialisation and are garbage after
 *     the call; the caller must not reuse it on another stream until this call's work is done.
 *   - Errors: every argument is validated before anything is launched. Status codes only; nothing
 *     throws across the boundary and nothing traps on the device.
 *       TP_ERR_INVALID_ARG  NULL required pointer, size out of range, bad metric/dtype/k, exclude_self
 *                           with N != M, output aliasing an input or another output (except the
 *                           documented dX/dY alias), misaligned pointer, workspace too small.
 *       TP_ERR_UNSUPPORTED  a valid request the library has no kernel for.
 *       TP_ERR_CUDA         a CUDA launch error (the runtime's error text is in tp_last_error()), or a
 *                           fault injected before launch (TP_FAULT_INJECT, see tp_device_status).
 *     Device-side conditions are not known when a call returns: the warps of the tensor-core kernels
 *     wait on one another with bounded waits (2 s), and a wait that gives up records a code in a
 *     per-device error word instead of trapping; tp_device_status reads it after the caller has
 *     synchronised (TP_ERR_TIMEOUT). There is no CPU fallback.
 *   - Backward outputs are written, not accumulated. A NULL gradient output means "not requested";
 *     its work is skipped. When X and Y are the same points (X == Y, N == M), dY may be the same
 *     pointer as dX: the sum dX + dY is then written there.
 *   - Results agree with an exact evaluation within floating tolerance, not bitwise: the sums run in
 *     a different order (the guide's "What to Check", precision). Top-k values and indices are exact
 *     whenever the scores are exact in the working precision.
 *   - Non-finite inputs are not supported; their results are unspecified.
 */
#ifndef TP_H_
#define TP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TP_OK = 0,
    TP_ERR_INVALID_ARG = 1,
    TP_ERR_UNSUPPORTED = 2,
    TP_ERR_CUDA = 3,
    TP_ERR_WORKSPACE = 4, /* reserved: a too-small workspace is reported as TP_ERR_INVALID_ARG */
    TP_ERR_TIMEOUT = 5    /* a bounded wait inside a kernel gave up (reported by tp_device_status) */
} tp_status;

typedef enum { TP_F32 = 0, TP_F64 = 1 } tp_dtype;

typedef enum { TP_SQEUCLIDEAN = 0, TP_LINEAR = 1, TP_RBF = 2 } tp_metric;

/* Pair masks, torchpairwise guide "Using Torchpairwise in Models", Score Expressions and Task Map
 * (tp.masks: causal, band, same_group). A masked pair leaves the consumer's reduction: it adds no term
 * to K@V, a log-sum-exp, a softmax or a displacement, top-k never selects it, and it gets no gradient.
 * A softmax row with every pair masked returns 0 (its log-sum-exp is -inf). TP_PAIRS_CAUSAL keeps
 * j <= i, TP_PAIRS_BAND keeps |i - j| <= band, TP_PAIRS_SAME_GROUP keeps row_group[i] ==
 * col_group[j]. These run in the streamed sweeps (the pages run them on materialised tiles). */
typedef enum { TP_PAIRS_ALL = 0, TP_PAIRS_CAUSAL = 1, TP_PAIRS_BAND = 2, TP_PAIRS_SAME_GROUP = 3 } tp_pair_mask;

/* The canonical score (see the file comment). Bias and weight pointers are device arrays of the
 * problem's dtype, [N] for rows and [M] for columns, or NULL when absent. gamma is used by TP_RBF
 * only. pair_mask selects a pair mask (above); band (>= 0) is read by TP_PAIRS_BAND only (any width of
 * N + M or more keeps every pair); row_group
 * [N] and col_group [M] are int32 device arrays read by TP_PAIRS_SAME_GROUP only (NULL otherwise). */
typedef struct {
    tp_metric metric;
    double gamma;
    double scale;
    int apply_exp;
    const void *row_bias, *col_bias, *row_weight, *col_weight;
    tp_pair_mask pair_mask;
    int64_t band;
    const int32_t *row_group, *col_group;
} tp_score;

/* The two point sets: X [N,D] and Y [M,D], device, row-major, contiguous. */
typedef struct {
    tp_dtype dtype;
    int64_t N, M, D;
    const void *X, *Y;
} tp_pairs;

/* ---------------------------------------------------------------------------------------------- */
/* forward consumers                                                                              */
/* ---------------------------------------------------------------------------------------------- */

/* Kernel product out_i = sum_j S_ij V_j, out [N,C].
 * Guide "Task Map", kernel attention / Nadaraya-Watson row: lazy(X, Y, "rbf", gamma) @ V; with
 * V = [V | ones] the last output column is the row mass sum_j S_ij. */
TP_API tp_status tp_pairwise_matmul(const tp_pairs* pairs, const tp_score* score, const void* V, int64_t C,
                             void* out, void* ws, size_t ws_bytes, void* stream);

/* Row log-sum-exp lse_i = log sum_j exp(S_ij), lse [N]; with exclude_self != 0 the pair j == i is
 * left out (requires N == M; a row with no pair left gives -inf).
 * Guide "Task Map", InfoNCE / NT-XEnt row (a log-sum-exp over the last axis with the self pair
 * excluded); "Score Expressions" example (the loss is minus the mean of the row log-sum-exp). */
TP_API tp_status tp_pairwise_logsumexp(const tp_pairs* pairs, const tp_score* score, int exclude_self,
                                void* lse, void* ws, size_t ws_bytes, void* stream);

/* Attention row out_i = sum_j softmax_j(S_ij) V_j, out [N,C]; also writes lse [N] (the row
 * log-sum-exp of S), which the backward takes back.
 * Guide introduction example and "Task Map", attention row: (lazy(Q, K, "linear") * s).softmax_matmul(V),
 * fused without a pair mask. */
TP_API tp_status tp_pairwise_softmax_matmul(const tp_pairs* pairs, const tp_score* score, const void* V,
                                     int64_t C, void* out, void* lse, void* ws, size_t ws_bytes,
                                     void* stream);

/* Displacement disp_i = sum_j S_ij (y_j - x_i), out [N,D].
 * Guide "Stein Variational Gradient Descent": the kernel's displacement method, which streams the
 * repulsive term sum_j k_ij (x_j - x_i). */
TP_API tp_status tp_pairwise_displacement(const tp_pairs* pairs, const tp_score* score, void* out, void* ws,
                                   size_t ws_bytes, void* stream);

/* SVGD direction phi_i = (1/n) sum_j k_ij (score_j - 2 gamma (x_j - x_i)), phi [n,D], with
 * k_ij = exp(-gamma |x_i - x_j|^2), n = M, in one sweep (one kernel evaluation per pair).
 * pairs->X and pairs->Y hold the particles (normally the same array, N == M); score [M,D] is the
 * target's score at each particle. Only gamma is read from the canonical score: the formula is the
 * bare rbf kernel.
 * Guide "Stein Variational Gradient Descent": phi = (K @ score - 2 gamma K.displacement()) / n. */
TP_API tp_status tp_svgd_direction(const tp_pairs* pairs, double gamma, const void* score, void* phi,
                            void* ws, size_t ws_bytes, void* stream);

/* Row top-k: the k smallest S_ij of each row (largest != 0: the k largest), values [N,k] and
 * indices [N,k] (int64), sorted by value (ascending; descending for largest) and, among equal
 * values, by ascending column index. 1 <= k <= min(M, 128). Under a pair mask a row with fewer than
 * k kept pairs fills its tail with value +inf (-inf for largest) and index -1.
 * Guide "Task Map", k-NN / retrieval row: lazy(X, R, "sqeuclidean").topk(k, largest=False), fused,
 * exact tie order; argmin and min are k = 1. */
TP_API tp_status tp_pairwise_topk(const tp_pairs* pairs, const tp_score* score, int k, int largest,
                           void* values, int64_t* indices, void* ws, size_t ws_bytes, void* stream);

/* The row log-sum-exp of tp_pairwise_logsumexp, for callers that cannot allocate device memory when
 * they need it: code running inside another allocator's critical section or out-of-memory callback,
 * real-time loops that forbid allocation after start-up, hosts that cannot size and own a workspace.
 * The guide has no counterpart to this entry point; it exists for those callers only.
 * There is no workspace argument: the scratch is a fixed 16 MiB array of device memory owned by this
 * library, held on every GPU that loads it until the process exits. A problem whose workspace
 * (tp_workspace_size("pairwise_logsumexp", ...)) exceeds 16 MiB is rejected with TP_ERR_INVALID_ARG
 * and a message in tp_last_error(), before anything is launched. Only fp32 with D = 64 (the
 * tensor-core path, which keeps an fp16 hi/lo copy of the points) can exceed it: beyond N = 54542 when
 * Y is X (the same array and count), or beyond N + M of about 55000 when they differ. Every other shape
 * needs at most 2 MiB.
 * The first call on a device looks up the array's address (with that device current); make that
 * first call before any stream capture. Every call shares the array and finds the previous call's
 * contents there; nothing in it needs clearing, but calls whose GPU work overlaps (different streams
 * or threads without ordering) race on it. Allocates nothing; every other convention, argument and
 * error is that of tp_pairwise_logsumexp. */
TP_API tp_status tp_pairwise_logsumexp_noalloc(const tp_pairs* pairs, const tp_score* score, int exclude_self,
                                               void* lse, void* stream);

/* ---------------------------------------------------------------------------------------------- */
/* backward by replay (torchpairwise guide, "Using Torchpairwise in Models", introduction)       */
/* Inputs are the forward's inputs plus the upstream gradient; outputs are gradients with the     */
/* shapes of X [N,D], Y [M,D], V [M,C], row bias/weight [N], column bias/weight [M]. A gradient   */
/* for a bias or weight that the score does not have must be NULL.                                */
/* ---------------------------------------------------------------------------------------------- */

/* Gradients of L = sum_ic grad_out_ic out_ic for out = tp_pairwise_matmul(...); grad_out [N,C]. */
TP_API tp_status tp_pairwise_matmul_backward(const tp_pairs* pairs, const tp_score* score, const void* V,
                                      int64_t C, const void* grad_out, void* dX, void* dY, void* dV,
                                      void* d_row_bias, void* d_col_bias, void* d_row_weight,
                                      void* d_col_weight, void* ws, size_t ws_bytes, void* stream);

/* Gradients of L = sum_i grad_lse_i lse_i; lse [N] is the forward's output, grad_lse [N]. */
TP_API tp_status tp_pairwise_logsumexp_backward(const tp_pairs* pairs, const tp_score* score,
                                         int exclude_self, const void* lse, const void* grad_lse,
                                         void* dX, void* dY, void* d_row_bias, void* d_col_bias,
                                         void* d_row_weight, void* d_col_weight, void* ws,
                                         size_t ws_bytes, void* stream);

/* Gradients of L = sum_ic grad_out_ic out_ic for out = tp_pairwise_softmax_matmul(...); out [N,C]
 * and lse [N] are the forward's outputs, grad_out [N,C]. */
TP_API tp_status tp_pairwise_softmax_matmul_backward(const tp_pairs* pairs, const tp_score* score,
                                              const void* V, int64_t C, const void* out,
                                              const void* lse, const void* grad_out, void* dX,
                                              void* dY, void* dV, void* d_row_bias,
                                              void* d_col_bias, void* d_row_weight,
                                              void* d_col_weight, void* ws, size_t ws_bytes,
                                              void* stream);

/* Gradients of L = sum_id grad_out_id disp_id for disp = tp_pairwise_displacement(...);
 * grad_out [N,D]. */
TP_API tp_status tp_pairwise_displacement_backward(const tp_pairs* pairs, const tp_score* score,
                                            const void* grad_out, void* dX, void* dY,
                                            void* d_row_bias, void* d_col_bias, void* d_row_weight,
                                            void* d_col_weight, void* ws, size_t ws_bytes,
                                            void* stream);

/* Gradients of L = sum_it grad_values_it values_it, through the selected pairs only (guide "What to
 * Check": selections route gradients through the selected pairs, not the indices). indices [N,k]
 * as returned by tp_pairwise_topk (each in [0, M)); grad_values [N,k]. Column gradients are
 * gathered per column in a deterministic order, without atomics. */
TP_API tp_status tp_pairwise_topk_backward(const tp_pairs* pairs, const tp_score* score, int k,
                                    const int64_t* indices, const void* grad_values, void* dX,
                                    void* dY, void* d_row_bias, void* d_col_bias,
                                    void* d_row_weight, void* d_col_weight, void* ws,
                                    size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------- */
/* helpers                                                                                        */
/* ---------------------------------------------------------------------------------------------- */

/* Workspace bytes an entry point needs for these shapes. `entry` is the entry point's name without
 * the "tp_" prefix, e.g. "pairwise_logsumexp_backward" or "svgd_direction"; C is V's width (ignored
 * where there is no V) and k the top-k size (ignored elsewhere). Returns (size_t)-1 for an unknown
 * entry or invalid sizes. Depends on the shapes only, never on the device. */
TP_API size_t tp_workspace_size(const char* entry, const tp_pairs* pairs, int64_t C, int k);

/* Static text for a status code. */
TP_API const char* tp_status_string(tp_status status);

/* Text of the last TP_ERR_* reported by this thread (argument name, CUDA error string). */
TP_API const char* tp_last_error(void);

/* Number of kernels enqueued by this thread since the counter was last reset (instrumentation for
 * launch counting; reset = 1 zeroes it and returns the previous value). */
TP_API int64_t tp_launch_count(int reset);

/* Instrumentation hook. When set, hook(kernel, phase, stream, user) is called on the host, on the
 * launching thread, immediately before (phase 0) and after (phase 1) every kernel launch this library
 * makes; `kernel` is a static name such as "bwd_sweep_lse_row" and `stream` the launch stream.
 * A profiler can record CUDA events there to time each kernel inside a real call sequence.
 * NULL removes the hook. Not thread-safe with respect to concurrent launches: set it while no other
 * thread is calling into libtp. */
typedef void (*tp_launch_hook)(const char* kernel, int phase, void* stream, void* user);
TP_API void tp_set_launch_hook(tp_launch_hook hook, void* user);

/* Kernel timer: per-launch device durations with no host callback in the launch path.
 * tp_timer_start(capacity) creates (or reuses) 2 * capacity CUDA events on the current device and
 * starts recording: immediately before and after every kernel launch this library makes, one event is
 * recorded on the launch stream (the host cost is the two cudaEventRecord calls). Launches beyond
 * `capacity` are not timed. Returns TP_ERR_INVALID_ARG for capacity < 1, TP_ERR_CUDA if events cannot
 * be created.
 * tp_timer_stop() stops recording and returns the number of launches timed.
 * tp_timer_read(i, &kernel, &ms) waits for the i-th timed launch (0-based, launch order) to complete,
 * then stores its static kernel name and its duration in milliseconds. Returns TP_ERR_INVALID_ARG for
 * an index outside the last recording, TP_ERR_CUDA if the events cannot be read.
 * Process-wide: start and stop it while no other thread is calling into libtp. The events stay owned by
 * the library (released at process exit). */
TP_API tp_status tp_timer_start(int64_t capacity);
TP_API int64_t tp_timer_stop(void);
TP_API tp_status tp_timer_read(int64_t index, const char** kernel, float* ms);

/* Device-side status of the current device: TP_OK, or TP_ERR_TIMEOUT when a bounded wait inside one of
 * this library's kernels gave up since the word was last reset (the message in tp_last_error() names the
 * kernel and the wait's site code). The results of the call whose kernel gave up are invalid. The word is
 * one per device and sticky: every kernel on every stream writes the same word, and the first code is
 * kept until reset != 0 clears it. The read is synchronous (cudaMemcpy on the legacy default stream);
 * call it after synchronising the streams whose work it should cover. TP_ERR_CUDA if the word cannot be
 * read. The first call of any entry point on a device looks up the word's address (with that device
 * current); make it before any stream capture.
 * The method's "What to Check" section (torchpairwise guide) has solvers report a status beside their
 * result; this is that convention for device-side waits.
 * Host-side fault injection for tests: with TP_FAULT_INJECT=<entry> in the environment (the entry point's
 * name without "tp_", e.g. "pairwise_logsumexp"), that entry returns TP_ERR_CUDA after validating its
 * arguments and before launching anything. The variable is read on every call. */
TP_API tp_status tp_device_status(int reset);

/* Self-test of the device-side status path: launches on `stream` one block whose single mbarrier wait
 * expects an arrival that never comes, bounded by limit_ns (1000 to 2e9 ns); the wait gives up, records
 * its code in the error word and the kernel returns. Nothing else is in flight in that kernel (no copy,
 * no tensor-core operation, no tensor memory), so giving up leaves the device usable. A following
 * tp_device_status (after synchronising) reports TP_ERR_TIMEOUT. TP_ERR_INVALID_ARG for a limit outside
 * the range. The guide has no counterpart; it exists to test the convention above. */
TP_API tp_status tp_selftest_bounded_wait(int64_t limit_ns, void* stream);

/* Self-test of the fp64 exponential every fp64 kernel of this library evaluates (a table-driven method:
 * "Stein Variational Gradient Descent" needs one fp64 exp per pair, and there is no fp64 special-function
 * unit): y[i] = exp(x[i]) for n doubles, device arrays, enqueued on `stream`. Its error is at most about
 * 1.2 ulp for x in [-707, 709.78]; below -707 it returns 0, above 709.78 +inf; NaN is not handled.
 * TP_ERR_INVALID_ARG for n < 0 or a NULL array with n > 0. The guide has no counterpart; it exists so the
 * routine can be tested against a reference exp. */
TP_API tp_status tp_selftest_exp64(const double* x, double* y, int64_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TP_H_ */
