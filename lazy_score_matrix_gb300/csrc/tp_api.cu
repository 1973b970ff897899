// The C-ABI of libtp (declared in include/tp.h): argument validation, split planning, workspace
// sizing and dispatch to the compiled kernel buckets. No kernel is compiled in this translation
// unit; every launcher is explicitly instantiated in an inst_*.cu file.
//
// Method: torchpairwise guide "Using Torchpairwise in Models" (introduction, "Task Map", "Score
// Expressions", "Stein Variational Gradient Descent").
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <string>
#include <type_traits>
#include <utility>
#include <vector>

#include "tp.h"
#include "tp_launch.h"

using namespace tp;

namespace tp {
size_t lse_tc_workspace(int64_t N, int64_t M, bool same);                  // tp_tc_lse.cu
int launch_lse_tc(const SweepArgs& a, void* lse, bool same, cudaStream_t s);  // tp_tc_lse.cu
size_t lse_bwd_tc_workspace(int64_t N);                                       // tp_tc_lse.cu
int launch_lse_bwd_sym_tc(const SweepArgs& a, cudaStream_t s);                // tp_tc_lse.cu
size_t topk_tc_workspace(int64_t N, int64_t M, int D, int k, bool same);                        // tp_tc_topk.cu
int launch_topk_tc(const SweepArgs& a, void* values, int64_t* indices, bool same, cudaStream_t s);  // tp_tc_topk.cu
size_t attn_tc_workspace(int64_t N, int64_t M, bool backward);                  // tp_tc_attn.cu
int launch_attn_fwd_tc(const AttnTcArgs& a, cudaStream_t s);                    // tp_tc_attn.cu
int launch_attn_bwd_tc(const AttnTcArgs& a, cudaStream_t s);                    // tp_tc_attn.cu
}  // namespace tp

namespace tp {
tp_status launched(int n);
tp_status injected_fault(const char* entry);  // tp_status.cu: TP_FAULT_INJECT
}  // namespace tp

namespace {

thread_local std::string g_err;
thread_local int64_t g_launches = 0;
tp_launch_hook g_hook = nullptr;
void* g_hook_user = nullptr;

// kernel timer (tp_timer_*): an event pair per launch, recorded from the launch path
struct KernelTimer {
    std::vector<cudaEvent_t> ev;     // 2 per slot
    std::vector<const char*> name;   // per slot
    int device = -1;
    int64_t capacity = 0, count = 0, recorded = 0;
    bool on = false;
};
KernelTimer g_timer;

tp_status fail(tp_status s, const std::string& msg) {
    g_err = msg;
    return s;
}

// Split heuristic of the streamed sweeps (part of the workspace size, so from the shapes only, never the
// device): enough CTAs for a GB300's 152 SMs at ~4 resident 128-thread CTAs each.
constexpr int64_t kTargetCtas = 152 * 4;
constexpr int kMaxSplits = 64;
constexpr size_t kAlign = 256;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Plan {
    int splits;
    int64_t cps;
};

// Deterministic split of the streamed set, from the shapes only: enough CTAs to fill the GPU,
// each split at least two tiles long.
Plan plan_split(int64_t nP, int64_t nQ) {
    const int64_t rowblocks = cdiv(nP, kThreads);
    const int64_t tiles = cdiv(nQ, kTile);
    int64_t s = cdiv(kTargetCtas, rowblocks);
    s = std::min<int64_t>(s, std::max<int64_t>(1, tiles / 2));
    s = std::min<int64_t>(s, kMaxSplits);
    s = std::max<int64_t>(s, 1);
    const int64_t cps = cdiv(tiles, s) * kTile;
    return Plan{(int)cdiv(nQ, cps), cps};
}

size_t esize(tp_dtype t) { return t == TP_F64 ? 8 : 4; }

// X and Y are the same points: one pointer AND one count. A caller may pass Y = Z and X = Z[:N] with
// N < M (the same pointer, fewer rows); the tensor-core paths then must not treat the two as one set,
// since a workspace copy of X holds only N rows.
bool same_points(const tp_pairs* p) { return p->X == p->Y && p->N == p->M; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Span {
    const void* p;
    size_t bytes;
    const char* name;
};

bool overlap(const Span& a, const Span& b) {
    if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// outputs must not overlap inputs or each other; `allow` lists output pairs that may coincide
tp_status check_alias(const std::vector<Span>& in, const std::vector<Span>& out,
                      std::pair<const void*, const void*> allow = {nullptr, nullptr}) {
    for (size_t o = 0; o < out.size(); ++o) {
        for (const Span& i : in)
            if (overlap(out[o], i))
                return fail(TP_ERR_INVALID_ARG, std::string(out[o].name) + " overlaps input " + i.name);
        for (size_t o2 = o + 1; o2 < out.size(); ++o2) {
            if (out[o].p && out[o].p == out[o2].p && out[o].p == allow.first && allow.first == allow.second) continue;
            if (overlap(out[o], out[o2]))
                return fail(TP_ERR_INVALID_ARG, std::string(out[o].name) + " overlaps output " + out[o2].name);
        }
    }
    return TP_OK;
}

tp_status check_pairs(const tp_pairs* p) {
    if (!p) return fail(TP_ERR_INVALID_ARG, "pairs is NULL");
    if (p->dtype != TP_F32 && p->dtype != TP_F64) return fail(TP_ERR_INVALID_ARG, "dtype must be TP_F32 or TP_F64");
    if (p->N < 1 || p->M < 1) return fail(TP_ERR_INVALID_ARG, "N and M must be >= 1");
    if (p->N >= (int64_t(1) << 31) || p->M >= (int64_t(1) << 31))
        return fail(TP_ERR_INVALID_ARG, "N and M must be below 2^31");
    if (p->D < 1 || p->D > 64) return fail(TP_ERR_INVALID_ARG, "D must be in [1, 64]");
    if (!p->X || !p->Y) return fail(TP_ERR_INVALID_ARG, "X and Y must be device pointers");
    const size_t es = esize(p->dtype);
    if (!aligned(p->X, es) || !aligned(p->Y, es)) return fail(TP_ERR_INVALID_ARG, "X/Y not aligned to the element size");
    return TP_OK;
}

tp_status check_score(const tp_score* s, const tp_pairs* p) {
    if (!s) return fail(TP_ERR_INVALID_ARG, "score is NULL");
    if (s->metric != TP_SQEUCLIDEAN && s->metric != TP_LINEAR && s->metric != TP_RBF)
        return fail(TP_ERR_INVALID_ARG, "unknown metric");
    const size_t es = esize(p->dtype);
    for (const void* q : {s->row_bias, s->col_bias, s->row_weight, s->col_weight})
        if (q && !aligned(q, es)) return fail(TP_ERR_INVALID_ARG, "bias/weight not aligned to the element size");
    switch (s->pair_mask) {
        case TP_PAIRS_ALL:
        case TP_PAIRS_CAUSAL: break;
        case TP_PAIRS_BAND:
            if (s->band < 0) return fail(TP_ERR_INVALID_ARG, "band must be >= 0");
            break;
        case TP_PAIRS_SAME_GROUP:
            if (!s->row_group || !s->col_group) return fail(TP_ERR_INVALID_ARG, "same-group mask needs row_group and col_group");
            if (!aligned(s->row_group, 4) || !aligned(s->col_group, 4))
                return fail(TP_ERR_INVALID_ARG, "row_group/col_group not aligned to 4 bytes");
            break;
        default: return fail(TP_ERR_INVALID_ARG, "unknown pair mask");
    }
    return TP_OK;
}

// The band width the kernels read: a width of N + M or more keeps every pair, so wider ones are read as
// N + M (the tensor-core schedule adds the width to point indices in 64-bit arithmetic).
int64_t pair_band(const tp_score* s, const tp_pairs* p) {
    const int64_t all = p->N + p->M;
    return s->band < all ? s->band : all;
}

tp_status check_C(int64_t C, const void* V) {
    if (C < 1 || C > 64) return fail(TP_ERR_INVALID_ARG, "C must be in [1, 64]");
    if (!V) return fail(TP_ERR_INVALID_ARG, "V is NULL");
    return TP_OK;
}

tp_status check_ptr(const void* p, const char* name, size_t es) {
    if (!p) return fail(TP_ERR_INVALID_ARG, std::string(name) + " is NULL");
    if (!aligned(p, es)) return fail(TP_ERR_INVALID_ARG, std::string(name) + " not aligned to the element size");
    return TP_OK;
}

tp_status check_ws(const void* ws, size_t have, size_t need) {
    if (need == 0) return TP_OK;
    if (!ws) return fail(TP_ERR_INVALID_ARG, "workspace is NULL but " + std::to_string(need) + " bytes are needed");
    if (have < need)
        return fail(TP_ERR_INVALID_ARG, "workspace too small: " + std::to_string(have) + " < " + std::to_string(need));
    if (!aligned(ws, kAlign)) return fail(TP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    return TP_OK;
}

std::vector<Span> score_spans(const tp_score* s, const tp_pairs* p) {
    const size_t es = esize(p->dtype);
    const bool groups = s->pair_mask == TP_PAIRS_SAME_GROUP;
    return {{s->row_bias, p->N * es, "row_bias"},
            {s->col_bias, p->M * es, "col_bias"},
            {s->row_weight, p->N * es, "row_weight"},
            {s->col_weight, p->M * es, "col_weight"},
            {groups ? s->row_group : nullptr, (size_t)p->N * 4, "row_group"},
            {groups ? s->col_group : nullptr, (size_t)p->M * 4, "col_group"}};
}

// Row-side (P = X) or column-side (P = Y) arguments of a sweep.
SweepArgs side_args(const tp_pairs* p, const tp_score* s, bool col) {
    SweepArgs a;
    std::memset(&a, 0, sizeof a);
    a.P = col ? p->Y : p->X;
    a.Q = col ? p->X : p->Y;
    a.nP = col ? p->M : p->N;
    a.nQ = col ? p->N : p->M;
    a.D = (int)p->D;
    a.metric = s->metric;
    a.gamma = s->gamma;
    a.scale = s->scale;
    a.apply_exp = s->apply_exp ? 1 : 0;
    a.pb = col ? s->col_bias : s->row_bias;
    a.qb = col ? s->row_bias : s->col_bias;
    a.pw = col ? s->col_weight : s->row_weight;
    a.qw = col ? s->row_weight : s->col_weight;
    a.affine = (s->row_bias || s->col_bias || s->row_weight || s->col_weight) ? 1 : 0;
    a.pm = (int)s->pair_mask;
    a.pcol = col ? 1 : 0;
    a.band = pair_band(s, p);
    if (s->pair_mask == TP_PAIRS_SAME_GROUP) {
        a.pg = col ? s->col_group : s->row_group;
        a.qg = col ? s->row_group : s->col_group;
    }
    const Plan pl = plan_split(a.nP, a.nQ);
    a.splits = pl.splits;
    a.cps = pl.cps;
    a.vecQ = (pad_bucket(a.D) == a.D && aligned(a.Q, 16)) ? 1 : 0;
    return a;
}

// TP_FORCE_SIMT=1 in the environment routes every call to the SIMT kernels (A/B comparisons).
bool force_simt() {
    static const bool v = [] {
        const char* e = getenv("TP_FORCE_SIMT");
        return e && e[0] && e[0] != '0';
    }();
    return v;
}

// The tensor-core symmetric backward (fp32, D = 64, X = Y, no row/column parameters) and the
// tensor-core top-k (fp32, D <= 64, k <= 32): both pass every parity test on the GPU and are several
// times faster than the SIMT sweeps they replace on the InfoNCE and k-NN workloads.
constexpr bool kTcBackward = true;
constexpr bool kTcTopk = true;

// The tensor-core log-sum-exp covers fp32, D = 64, no row/column parameters, 16-byte aligned points.
bool lse_tc_shape(const tp_pairs* p) { return p->dtype == TP_F32 && p->D == 64; }
bool lse_tc_eligible(const tp_pairs* p, const tp_score* s) {
    return !force_simt() && lse_tc_shape(p) && !s->row_bias && !s->col_bias && !s->row_weight && !s->col_weight &&
           s->pair_mask == TP_PAIRS_ALL && aligned(p->X, 16) && aligned(p->Y, 16);
}

// Tensor-core attention: softmax_matmul and its backward for fp32, D = C = 64, a linear score without
// exp or row/column parameters, 16-byte aligned rows, no pair mask or an index mask (causal, band: the
// epilogues test the pair's indices; same-group masks stay on the streamed sweeps).
constexpr bool kTcAttention = true;
bool attn_tc_shape(const tp_pairs* p, int64_t C) { return p->dtype == TP_F32 && p->D == 64 && C == 64; }
bool attn_tc_eligible(const tp_pairs* p, const tp_score* s, int64_t C, std::initializer_list<const void*> rows) {
    if (!kTcAttention || force_simt() || !attn_tc_shape(p, C) || s->metric != TP_LINEAR || s->apply_exp || s->row_bias ||
        s->col_bias || s->row_weight || s->col_weight || s->pair_mask == TP_PAIRS_SAME_GROUP || !aligned(p->X, 16) ||
        !aligned(p->Y, 16))
        return false;
    for (const void* q : rows)
        if (q && !aligned(q, 16)) return false;
    return true;
}

// The tensor-core top-k covers fp32, D <= 64, k <= 32, no row/column parameters.
bool topk_tc_shape(const tp_pairs* p, int k) { return p->dtype == TP_F32 && p->D <= 64 && k >= 1 && k <= kTopkMax; }
bool topk_tc_eligible(const tp_pairs* p, const tp_score* s, int k) {
    return kTcTopk && !force_simt() && topk_tc_shape(p, k) && !s->row_bias && !s->col_bias && !s->row_weight &&
           !s->col_weight && s->pair_mask == TP_PAIRS_ALL;
}

// A tensor-core launcher's result: kernels launched, or -1 (a TMA tensor map could not be encoded), or -3
// (the device error word could not be looked up; the reason is already in tp_last_error).
tp_status tc_launched(int n) {
    if (n == -3) return TP_ERR_CUDA;
    if (n < 0) return fail(TP_ERR_CUDA, "could not encode the TMA tensor maps (cuTensorMapEncodeTiled)");
    return launched(n);
}

template <int V>
using IC = std::integral_constant<int, V>;

template <class F>
void with_dp(int dp, F&& f) {
    switch (dp) {
        case 4: f(IC<4>{}); break;
        case 8: f(IC<8>{}); break;
        case 16: f(IC<16>{}); break;
        case 32: f(IC<32>{}); break;
        default: f(IC<64>{}); break;
    }
}
template <class F>
void with_cp(int cp, F&& f) {
    switch (cp) {
        case 4: f(IC<4>{}); break;
        case 16: f(IC<16>{}); break;
        default: f(IC<64>{}); break;
    }
}
template <class F>
void with_k(int k, F&& f) {
    switch (k) {
        case 1: f(IC<1>{}); break;
        case 4: f(IC<4>{}); break;
        case 8: f(IC<8>{}); break;
        case 16: f(IC<16>{}); break;
        default: f(IC<32>{}); break;
    }
}

// forward sweep + merge for the value-carrying modes (matmul, softmax): DP x CP x affine
template <class T, int MODE>
int run_fwd_vals(const SweepArgs& a, cudaStream_t st) {
    with_dp(pad_bucket(a.D), [&](auto dp) {
        with_cp(cpad_bucket(a.C), [&](auto cp) {
            if (a.affine) launch_fwd<T, decltype(dp)::value, decltype(cp)::value, MODE, true>(a, st);
            else launch_fwd<T, decltype(dp)::value, decltype(cp)::value, MODE, false>(a, st);
        });
    });
    if (a.splits > 1) {
        launch_fwd_merge<T, MODE>(a, st);
        return 2;
    }
    return 1;
}

// forward sweep + merge for lse / displacement (DP x affine) and svgd (DP)
template <class T, int MODE>
int run_fwd_plain(const SweepArgs& a, cudaStream_t st) {
    with_dp(pad_bucket(a.D), [&](auto dp) {
        if constexpr (MODE == kSvgd) launch_fwd<T, decltype(dp)::value, 4, MODE, false>(a, st);
        else if (a.affine) launch_fwd<T, decltype(dp)::value, 4, MODE, true>(a, st);
        else launch_fwd<T, decltype(dp)::value, 4, MODE, false>(a, st);
    });
    if (a.splits > 1) {
        launch_fwd_merge<T, MODE>(a, st);
        return 2;
    }
    return 1;
}

// workspace bytes of one sweep's partial states
size_t partial_bytes(const SweepArgs& a, int width, size_t es) {
    return a.splits > 1 ? align_up((size_t)a.splits * width * a.nP * es) : 0;
}

int fwd_width(int mode, int D, int C) {
    switch (mode) {
        case kMatmul: return C;
        case kSoftmax: return 2 + C;
        case kLse: return 2;
        default: return D + 1;  // kDisp, kSvgd: D sums and the row mass
    }
}

// widths of the backward partial states (must match bwd_state_width in the kernels)
int bwd_width(int mode, int side, bool g, bool v, int D, int C) {
    int w = 0;
    if (g) {
        w += D + 3;
        if (mode == kBDisp) w += side == kRow ? 1 : D;
    }
    if (v) w += C;
    return w;
}

// Largest workspace any sweep of a backward entry needs (sweeps run one after another on the
// stream and reuse the same region); `extra` bytes in front (softmax delta).
size_t bwd_ws(const tp_pairs* p, int mode, int64_t C, size_t extra) {
    const size_t es = esize(p->dtype);
    tp_score s;
    std::memset(&s, 0, sizeof s);
    s.metric = TP_LINEAR;
    const SweepArgs r = side_args(p, &s, false), c = side_args(p, &s, true);
    const int D = (int)p->D, Ci = (int)C;
    size_t need = partial_bytes(r, bwd_width(mode, kRow, true, false, D, Ci), es);
    need = std::max(need, partial_bytes(c, bwd_width(mode, kCol, true, mode == kBMatmul || mode == kBSoftmax, D, Ci), es));
    return extra + need;
}

size_t ws_size(const char* entry, const tp_pairs* p, int64_t C, int k) {
    if (!entry || !p || p->N < 1 || p->M < 1 || p->D < 1 || p->D > 64 || (p->dtype != TP_F32 && p->dtype != TP_F64))
        return (size_t)-1;
    const size_t es = esize(p->dtype);
    tp_score s;
    std::memset(&s, 0, sizeof s);
    s.metric = TP_LINEAR;
    const SweepArgs r = side_args(p, &s, false);
    const std::string e(entry);
    const int D = (int)p->D;
    const bool needC = e.find("matmul") != std::string::npos;
    if (needC && (C < 1 || C > 64)) return (size_t)-1;
    if (e == "pairwise_matmul") return partial_bytes(r, fwd_width(kMatmul, D, (int)C), es);
    if (e == "pairwise_softmax_matmul") {
        const size_t simt = partial_bytes(r, fwd_width(kSoftmax, D, (int)C), es);
        if (!(kTcAttention && attn_tc_shape(p, C))) return simt;
        return std::max(simt, lse_tc_workspace(p->N, p->M, same_points(p)) +
                                  attn_tc_workspace(p->N, p->M, false));
    }
    if (e == "pairwise_logsumexp") {
        const size_t simt = partial_bytes(r, fwd_width(kLse, D, 0), es);
        return lse_tc_shape(p) ? std::max(simt, lse_tc_workspace(p->N, p->M, same_points(p))) : simt;
    }
    if (e == "pairwise_displacement") return partial_bytes(r, fwd_width(kDisp, D, 0), es);
    if (e == "svgd_direction") return partial_bytes(r, fwd_width(kSvgd, D, 0), es);
    if (e == "pairwise_topk") {
        if (k < 1 || k > p->M || k > kTopkMax) return (size_t)-1;
        const int K = topk_bucket(k);
        const size_t simt = r.splits > 1 ? align_up((size_t)r.splits * K * r.nP * (es + 4)) : 0;
        return kTcTopk && topk_tc_shape(p, k) ? std::max(simt, topk_tc_workspace(p->N, p->M, D, k, same_points(p))) : simt;
    }
    if (e == "pairwise_matmul_backward") return bwd_ws(p, kBMatmul, C, 0);
    if (e == "pairwise_softmax_matmul_backward") {
        const size_t simt = bwd_ws(p, kBSoftmax, C, align_up(p->N * es));
        return kTcAttention && attn_tc_shape(p, C) ? std::max(simt, attn_tc_workspace(p->N, p->M, true)) : simt;
    }
    if (e == "pairwise_logsumexp_backward") {
        const size_t simt = bwd_ws(p, kBLse, 0, 0);
        const bool sym = same_points(p);
        return kTcBackward && lse_tc_shape(p) && sym ? std::max(simt, lse_bwd_tc_workspace(p->N)) : simt;
    }
    if (e == "pairwise_displacement_backward") return bwd_ws(p, kBDisp, 0, 0);
    if (e == "pairwise_topk_backward") {
        if (k < 1 || k > p->M) return (size_t)-1;
        return align_up(p->M * 4) * 3 + align_up(4) + align_up((size_t)p->N * k * 4);
    }
    return (size_t)-1;
}

// dispatch on the dtype
template <class F>
tp_status by_dtype(tp_dtype t, F&& f) {
    if (t == TP_F32) return f(float{});
    return f(double{});
}

// --- the softmax backward's row pre-pass: delta_i = dO_i . out_i -------------------------------
template <class T>
__global__ void softmax_delta_kernel(const T* __restrict__ dO, const T* __restrict__ out, int64_t N, int C,
                                     T* __restrict__ delta) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N) return;
    T acc = T(0);
    for (int c = 0; c < C; ++c) acc = fma(dO[i * C + c], out[i * C + c], acc);
    delta[i] = acc;
}

}  // namespace

// ---------------------------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------------------------

namespace {

struct Grads {
    void *dX, *dY, *dV, *dbr, *dbc, *dwr, *dwc;
};

tp_status check_grads(const tp_pairs* pr, const tp_score* sc, const Grads& g, int64_t C, std::vector<Span> in,
                      void* ws, size_t ws_bytes) {
    const size_t es = esize(pr->dtype);
    for (void* q : {g.dX, g.dY, g.dV, g.dbr, g.dbc, g.dwr, g.dwc})
        if (q && !aligned(q, es)) return fail(TP_ERR_INVALID_ARG, "gradient output not aligned to the element size");
    if (g.dbr && !sc->row_bias) return fail(TP_ERR_INVALID_ARG, "d_row_bias given but the score has no row bias");
    if (g.dbc && !sc->col_bias) return fail(TP_ERR_INVALID_ARG, "d_col_bias given but the score has no column bias");
    if (g.dwr && !sc->row_weight) return fail(TP_ERR_INVALID_ARG, "d_row_weight given but the score has no row weight");
    if (g.dwc && !sc->col_weight)
        return fail(TP_ERR_INVALID_ARG, "d_col_weight given but the score has no column weight");
    const bool same = g.dX && g.dX == g.dY;
    if (same && !same_points(pr))
        return fail(TP_ERR_INVALID_ARG, "dX and dY may only coincide when X and Y are the same points");
    std::vector<Span> sp = score_spans(sc, pr);
    in.insert(in.end(), sp.begin(), sp.end());
    in.push_back({pr->X, pr->N * pr->D * es, "X"});
    in.push_back({pr->Y, pr->M * pr->D * es, "Y"});
    return check_alias(in,
                       {{g.dX, pr->N * pr->D * es, "dX"},
                        {g.dY, pr->M * pr->D * es, "dY"},
                        {g.dV, pr->M * C * es, "dV"},
                        {g.dbr, pr->N * es, "d_row_bias"},
                        {g.dbc, pr->M * es, "d_col_bias"},
                        {g.dwr, pr->N * es, "d_row_weight"},
                        {g.dwc, pr->M * es, "d_col_weight"},
                        {ws, ws_bytes, "ws"}},
                       {g.dX, g.dY});
}

// One backward sweep (+ merge) for compile-time buckets.
template <class T, int DP, int CP, int MODE, int SIDE, bool G, bool V>
int bwd_step(const SweepArgs& a, cudaStream_t st) {
    launch_bwd<T, DP, CP, MODE, SIDE, G, V>(a, st);
    if (a.splits > 1) {
        launch_bwd_merge<T, MODE, SIDE, G, V>(a, st);
        return 2;
    }
    return 1;
}

// Row sweep then column sweep(s) of a backward entry for one (DP, CP) bucket. `row` / `col` are
// filled in except for the gradient outputs, which come from g.
template <class T, int MODE, int DP, int CP>
int run_backward_t(SweepArgs row, SweepArgs col, const Grads& g, cudaStream_t st) {
    constexpr bool VALS = MODE == kBMatmul || MODE == kBSoftmax;
    int n = 0;
    row.gP = g.dX;
    row.gPb = g.dbr;
    row.gPw = g.dwr;
    if (row.gP || row.gPb || row.gPw) n += bwd_step<T, DP, CP, MODE, kRow, true, false>(row, st);
    col.gP = g.dY;
    col.gPb = g.dbc;
    col.gPw = g.dwc;
    col.gV = g.dV;
    col.accumulate = (g.dY && g.dY == g.dX) ? 1 : 0;
    const bool need_g = col.gP || col.gPb || col.gPw;
    const bool need_v = VALS && col.gV;
    if constexpr (VALS) {
        if constexpr (fused_col_sweep(DP, CP)) {
            if (need_g || need_v) n += bwd_step<T, DP, CP, MODE, kCol, true, true>(col, st);
        } else {
            if (need_g) {
                SweepArgs c1 = col;
                c1.gV = nullptr;
                n += bwd_step<T, DP, CP, MODE, kCol, true, false>(c1, st);
            }
            if (need_v) {
                SweepArgs c2 = col;
                c2.gP = c2.gPb = c2.gPw = nullptr;
                n += bwd_step<T, DP, CP, MODE, kCol, false, true>(c2, st);
            }
        }
    } else {
        if (need_g) n += bwd_step<T, DP, CP, MODE, kCol, true, false>(col, st);
    }
    return n;
}

template <class T, int MODE>
int run_backward(const SweepArgs& row, const SweepArgs& col, const Grads& g, cudaStream_t st) {
    constexpr bool VALS = MODE == kBMatmul || MODE == kBSoftmax;
    int n = 0;
    with_dp(pad_bucket(row.D), [&](auto dp) {
        constexpr int DP = decltype(dp)::value;
        if constexpr (VALS) {
            with_cp(cpad_bucket(row.C), [&](auto c) { n = run_backward_t<T, MODE, DP, decltype(c)::value>(row, col, g, st); });
        } else {
            n = run_backward_t<T, MODE, DP, 4>(row, col, g, st);
        }
    });
    return n;
}

}  // namespace

namespace tp {
void set_last_error(const std::string& msg) { g_err = msg; }

tp_status launched(int n) {
    g_launches += n;
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(TP_ERR_CUDA, std::string("CUDA launch failed: ") + cudaGetErrorString(e));
    return TP_OK;
}

void launch_hook(const char* kernel, int phase, cudaStream_t s) {
    if (g_timer.on && g_timer.count < g_timer.capacity) {
        cudaEventRecord(g_timer.ev[2 * g_timer.count + phase], s);
        if (phase == 1) g_timer.name[g_timer.count++] = kernel;
    }
    if (g_hook) g_hook(kernel, phase, static_cast<void*>(s), g_hook_user);
}
}  // namespace tp

// ================================================================================================
// C ABI
// ================================================================================================

extern "C" {

const char* tp_status_string(tp_status s) {
    switch (s) {
        case TP_OK: return "TP_OK";
        case TP_ERR_INVALID_ARG: return "TP_ERR_INVALID_ARG: invalid argument";
        case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED: not supported by the library";
        case TP_ERR_CUDA: return "TP_ERR_CUDA: CUDA error";
        case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE: workspace error";
        case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT: device wait timed out";
    }
    return "unknown tp_status";
}

const char* tp_last_error(void) { return g_err.c_str(); }

void tp_set_launch_hook(tp_launch_hook hook, void* user) {
    g_hook = hook;
    g_hook_user = user;
}

tp_status tp_timer_start(int64_t capacity) {
    if (capacity < 1) return fail(TP_ERR_INVALID_ARG, "tp_timer_start: capacity must be >= 1");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(TP_ERR_CUDA, "tp_timer_start: no current device");
    if (dev != g_timer.device) {  // events belong to the device current at their creation
        for (cudaEvent_t e : g_timer.ev) cudaEventDestroy(e);
        g_timer.ev.clear();
        g_timer.device = dev;
    }
    while ((int64_t)g_timer.ev.size() < 2 * capacity) {
        cudaEvent_t e;
        const cudaError_t ce = cudaEventCreate(&e);
        if (ce != cudaSuccess) return fail(TP_ERR_CUDA, std::string("tp_timer_start: ") + cudaGetErrorString(ce));
        g_timer.ev.push_back(e);
    }
    g_timer.name.assign((size_t)capacity, nullptr);
    g_timer.capacity = capacity;
    g_timer.count = 0;
    g_timer.recorded = 0;
    g_timer.on = true;
    return TP_OK;
}

int64_t tp_timer_stop(void) {
    g_timer.on = false;
    g_timer.recorded = g_timer.count;
    return g_timer.recorded;
}

tp_status tp_timer_read(int64_t i, const char** kernel, float* ms) {
    if (i < 0 || i >= g_timer.recorded || !kernel || !ms)
        return fail(TP_ERR_INVALID_ARG, "tp_timer_read: index outside the last recording");
    cudaError_t ce = cudaEventSynchronize(g_timer.ev[2 * i + 1]);
    if (ce == cudaSuccess) ce = cudaEventElapsedTime(ms, g_timer.ev[2 * i], g_timer.ev[2 * i + 1]);
    if (ce != cudaSuccess) return fail(TP_ERR_CUDA, std::string("tp_timer_read: ") + cudaGetErrorString(ce));
    *kernel = g_timer.name[i];
    return TP_OK;
}

int64_t tp_launch_count(int reset) {
    const int64_t v = g_launches;
    if (reset) g_launches = 0;
    return v;
}

size_t tp_workspace_size(const char* entry, const tp_pairs* pairs, int64_t C, int k) {
    return ws_size(entry, pairs, C, k);
}

#define TP_CHECK(expr)                    \
    do {                                  \
        const tp_status _st = (expr);     \
        if (_st != TP_OK) return _st;     \
    } while (0)

tp_status tp_pairwise_matmul(const tp_pairs* pr, const tp_score* sc, const void* V, int64_t C, void* out, void* ws,
                             size_t ws_bytes, void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    TP_CHECK(check_C(C, V));
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(V, "V", es));
    TP_CHECK(check_ptr(out, "out", es));
    std::vector<Span> in = score_spans(sc, pr);
    in.push_back({pr->X, pr->N * pr->D * es, "X"});
    in.push_back({pr->Y, pr->M * pr->D * es, "Y"});
    in.push_back({V, pr->M * C * es, "V"});
    TP_CHECK(check_alias(in, {{out, pr->N * C * es, "out"}, {ws, ws_bytes, "ws"}}));
    const size_t need = ws_size("pairwise_matmul", pr, C, 0);
    TP_CHECK(check_ws(ws, ws_bytes, need));
    SweepArgs a = side_args(pr, sc, false);
    a.C = (int)C;
    a.Vq = V;
    a.vecV = (cpad_bucket(a.C) == a.C && aligned(V, 16)) ? 1 : 0;
    a.out = out;
    a.ws = ws;
    TP_CHECK(injected_fault("pairwise_matmul"));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return by_dtype(pr->dtype, [&](auto t) {
        using T = decltype(t);
        return launched(run_fwd_vals<T, kMatmul>(a, st));
    });
}

tp_status tp_pairwise_logsumexp(const tp_pairs* pr, const tp_score* sc, int exclude_self, void* lse, void* ws,
                                size_t ws_bytes, void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(lse, "lse", es));
    if (exclude_self && pr->N != pr->M) return fail(TP_ERR_INVALID_ARG, "exclude_self needs N == M");
    std::vector<Span> in = score_spans(sc, pr);
    in.push_back({pr->X, pr->N * pr->D * es, "X"});
    in.push_back({pr->Y, pr->M * pr->D * es, "Y"});
    TP_CHECK(check_alias(in, {{lse, pr->N * es, "lse"}, {ws, ws_bytes, "ws"}}));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("pairwise_logsumexp", pr, 0, 0)));
    TP_CHECK(injected_fault("pairwise_logsumexp"));
    SweepArgs a = side_args(pr, sc, false);
    a.exclude_self = exclude_self ? 1 : 0;
    a.out = lse;
    a.ws = ws;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (lse_tc_eligible(pr, sc)) {
        return tc_launched(launch_lse_tc(a, lse, same_points(pr), st));
    }
    return by_dtype(pr->dtype, [&](auto t) { return launched(run_fwd_plain<decltype(t), kLse>(a, st)); });
}

tp_status tp_pairwise_softmax_matmul(const tp_pairs* pr, const tp_score* sc, const void* V, int64_t C, void* out,
                                     void* lse, void* ws, size_t ws_bytes, void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    TP_CHECK(check_C(C, V));
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(V, "V", es));
    TP_CHECK(check_ptr(out, "out", es));
    TP_CHECK(check_ptr(lse, "lse", es));
    std::vector<Span> in = score_spans(sc, pr);
    in.push_back({pr->X, pr->N * pr->D * es, "X"});
    in.push_back({pr->Y, pr->M * pr->D * es, "Y"});
    in.push_back({V, pr->M * C * es, "V"});
    TP_CHECK(check_alias(in, {{out, pr->N * C * es, "out"}, {lse, pr->N * es, "lse"}, {ws, ws_bytes, "ws"}}));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("pairwise_softmax_matmul", pr, C, 0)));
    TP_CHECK(injected_fault("pairwise_softmax_matmul"));
    SweepArgs a = side_args(pr, sc, false);
    a.C = (int)C;
    a.Vq = V;
    a.vecV = (cpad_bucket(a.C) == a.C && aligned(V, 16)) ? 1 : 0;
    a.out = out;
    a.out2 = lse;
    a.ws = ws;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (attn_tc_eligible(pr, sc, C, {V, out, lse})) {
        // one sweep with an online softmax writes out and lse
        const bool same = same_points(pr);
        const int n1 = 0;
        AttnTcArgs t{};
        t.Q = static_cast<const float*>(pr->X);
        t.K = static_cast<const float*>(pr->Y);
        t.V = static_cast<const float*>(V);
        t.N = pr->N;
        t.M = pr->M;
        t.scale = sc->scale;
        t.lse_out = static_cast<float*>(lse);
        t.out = static_cast<float*>(out);
        t.pm = (int)sc->pair_mask;
        t.band = pair_band(sc, pr);
        t.ws = static_cast<char*>(ws) + lse_tc_workspace(pr->N, pr->M, same);
        const int n2 = launch_attn_fwd_tc(t, st);
        if (n2 < 0) {
            launched(n1);
            return tc_launched(n2);
        }
        return launched(n1 + n2);
    }
    return by_dtype(pr->dtype, [&](auto t) { return launched(run_fwd_vals<decltype(t), kSoftmax>(a, st)); });
}

tp_status tp_pairwise_displacement(const tp_pairs* pr, const tp_score* sc, void* out, void* ws, size_t ws_bytes,
                                   void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(out, "out", es));
    std::vector<Span> in = score_spans(sc, pr);
    in.push_back({pr->X, pr->N * pr->D * es, "X"});
    in.push_back({pr->Y, pr->M * pr->D * es, "Y"});
    TP_CHECK(check_alias(in, {{out, pr->N * pr->D * es, "out"}, {ws, ws_bytes, "ws"}}));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("pairwise_displacement", pr, 0, 0)));
    TP_CHECK(injected_fault("pairwise_displacement"));
    SweepArgs a = side_args(pr, sc, false);
    a.out = out;
    a.ws = ws;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return by_dtype(pr->dtype, [&](auto t) { return launched(run_fwd_plain<decltype(t), kDisp>(a, st)); });
}

tp_status tp_svgd_direction(const tp_pairs* pr, double gamma, const void* score, void* phi, void* ws,
                            size_t ws_bytes, void* stream) {
    TP_CHECK(check_pairs(pr));
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(score, "score", es));
    TP_CHECK(check_ptr(phi, "phi", es));
    std::vector<Span> in = {{pr->X, pr->N * pr->D * es, "X"}, {pr->Y, pr->M * pr->D * es, "Y"},
                            {score, pr->M * pr->D * es, "score"}};
    TP_CHECK(check_alias(in, {{phi, pr->N * pr->D * es, "phi"}, {ws, ws_bytes, "ws"}}));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("svgd_direction", pr, 0, 0)));
    TP_CHECK(injected_fault("svgd_direction"));
    tp_score s;
    std::memset(&s, 0, sizeof s);
    s.metric = TP_RBF;
    s.gamma = gamma;
    s.scale = 1.0;
    SweepArgs a = side_args(pr, &s, false);
    a.Vq = score;
    a.vecV = a.vecQ && aligned(score, 16) ? 1 : 0;
    a.out = phi;
    a.ws = ws;
    a.inv_n = 1.0 / (double)pr->M;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return by_dtype(pr->dtype, [&](auto t) { return launched(run_fwd_plain<decltype(t), kSvgd>(a, st)); });
}

tp_status tp_pairwise_topk(const tp_pairs* pr, const tp_score* sc, int k, int largest, void* values,
                           int64_t* indices, void* ws, size_t ws_bytes, void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    if (k < 1 || k > pr->M || k > 128) return fail(TP_ERR_INVALID_ARG, "k must be in [1, min(M, 128)]");
    if (k > kTopkMax) return fail(TP_ERR_UNSUPPORTED, "k above 32 is not compiled into the library");
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(values, "values", es));
    TP_CHECK(check_ptr(indices, "indices", 8));
    std::vector<Span> in = score_spans(sc, pr);
    in.push_back({pr->X, pr->N * pr->D * es, "X"});
    in.push_back({pr->Y, pr->M * pr->D * es, "Y"});
    TP_CHECK(check_alias(in, {{values, (size_t)(pr->N * k) * es, "values"}, {indices, (size_t)(pr->N * k) * 8, "indices"},
                              {ws, ws_bytes, "ws"}}));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("pairwise_topk", pr, 0, k)));
    TP_CHECK(injected_fault("pairwise_topk"));
    SweepArgs a = side_args(pr, sc, false);
    a.k = k;
    a.largest = largest ? 1 : 0;
    a.out = values;
    a.out2 = indices;
    a.ws = ws;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (topk_tc_eligible(pr, sc, k)) {
        return tc_launched(launch_topk_tc(a, values, indices, same_points(pr), st));
    }
    return by_dtype(pr->dtype, [&](auto t) {
        using T = decltype(t);
        int n = 1;
        with_dp(pad_bucket(a.D), [&](auto dp) {
            with_k(topk_bucket(k), [&](auto kk) {
                if (a.affine) launch_topk<T, decltype(dp)::value, decltype(kk)::value, true>(a, st);
                else launch_topk<T, decltype(dp)::value, decltype(kk)::value, false>(a, st);
                if (a.splits > 1) {
                    launch_topk_merge<T, decltype(kk)::value>(a, st);
                    n = 2;
                }
            });
        });
        return launched(n);
    });
}


tp_status tp_pairwise_matmul_backward(const tp_pairs* pr, const tp_score* sc, const void* V, int64_t C,
                                      const void* grad_out, void* dX, void* dY, void* dV, void* d_row_bias,
                                      void* d_col_bias, void* d_row_weight, void* d_col_weight, void* ws,
                                      size_t ws_bytes, void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    TP_CHECK(check_C(C, V));
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(V, "V", es));
    TP_CHECK(check_ptr(grad_out, "grad_out", es));
    const Grads g{dX, dY, dV, d_row_bias, d_col_bias, d_row_weight, d_col_weight};
    TP_CHECK(check_grads(pr, sc, g, C, {{V, pr->M * C * es, "V"}, {grad_out, pr->N * C * es, "grad_out"}}, ws,
                         ws_bytes));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("pairwise_matmul_backward", pr, C, 0)));
    TP_CHECK(injected_fault("pairwise_matmul_backward"));
    SweepArgs row = side_args(pr, sc, false), col = side_args(pr, sc, true);
    row.C = col.C = (int)C;
    row.Vp = grad_out;
    row.Vq = V;
    row.vecV = (cpad_bucket(row.C) == row.C && aligned(V, 16)) ? 1 : 0;
    col.Vp = V;
    col.Vq = grad_out;
    col.vecV = (cpad_bucket(col.C) == col.C && aligned(grad_out, 16)) ? 1 : 0;
    row.ws = col.ws = ws;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return by_dtype(pr->dtype, [&](auto t) { return launched(run_backward<decltype(t), kBMatmul>(row, col, g, st)); });
}

tp_status tp_pairwise_logsumexp_backward(const tp_pairs* pr, const tp_score* sc, int exclude_self, const void* lse,
                                         const void* grad_lse, void* dX, void* dY, void* d_row_bias,
                                         void* d_col_bias, void* d_row_weight, void* d_col_weight, void* ws,
                                         size_t ws_bytes, void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    if (exclude_self && pr->N != pr->M) return fail(TP_ERR_INVALID_ARG, "exclude_self needs N == M");
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(lse, "lse", es));
    TP_CHECK(check_ptr(grad_lse, "grad_lse", es));
    const Grads g{dX, dY, nullptr, d_row_bias, d_col_bias, d_row_weight, d_col_weight};
    TP_CHECK(check_grads(pr, sc, g, 1, {{lse, pr->N * es, "lse"}, {grad_lse, pr->N * es, "grad_lse"}}, ws,
                         ws_bytes));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("pairwise_logsumexp_backward", pr, 0, 0)));
    TP_CHECK(injected_fault("pairwise_logsumexp_backward"));
    SweepArgs row = side_args(pr, sc, false), col = side_args(pr, sc, true);
    row.lse = col.lse = lse;
    row.glse = col.glse = grad_lse;
    row.exclude_self = col.exclude_self = exclude_self ? 1 : 0;
    row.ws = col.ws = ws;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Same points, summed gradient wanted, no row/column parameters: the score is symmetric and one
    // sweep gives sum_j (H_kj + H_jk) dt_kj/dz_k, each pair evaluated once.
    const bool symmetric = dX && dX == dY && same_points(pr) && !sc->row_bias && !sc->col_bias &&
                           !sc->row_weight && !sc->col_weight && sc->pair_mask == TP_PAIRS_ALL;
    if (symmetric) {
        row.gP = dX;
        if (kTcBackward && lse_tc_eligible(pr, sc)) {
            return tc_launched(launch_lse_bwd_sym_tc(row, st));
        }
        return by_dtype(pr->dtype, [&](auto t) {
            using T = decltype(t);
            int n = 0;
            with_dp(pad_bucket(row.D), [&](auto dp) { n = bwd_step<T, decltype(dp)::value, 4, kBLseSym, kRow, true, false>(row, st); });
            return launched(n);
        });
    }
    return by_dtype(pr->dtype, [&](auto t) { return launched(run_backward<decltype(t), kBLse>(row, col, g, st)); });
}

tp_status tp_pairwise_softmax_matmul_backward(const tp_pairs* pr, const tp_score* sc, const void* V, int64_t C,
                                              const void* out, const void* lse, const void* grad_out, void* dX,
                                              void* dY, void* dV, void* d_row_bias, void* d_col_bias,
                                              void* d_row_weight, void* d_col_weight, void* ws, size_t ws_bytes,
                                              void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    TP_CHECK(check_C(C, V));
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(V, "V", es));
    TP_CHECK(check_ptr(out, "out", es));
    TP_CHECK(check_ptr(lse, "lse", es));
    TP_CHECK(check_ptr(grad_out, "grad_out", es));
    const Grads g{dX, dY, dV, d_row_bias, d_col_bias, d_row_weight, d_col_weight};
    TP_CHECK(check_grads(pr, sc, g, C,
                         {{V, pr->M * C * es, "V"},
                          {out, pr->N * C * es, "out"},
                          {lse, pr->N * es, "lse"},
                          {grad_out, pr->N * C * es, "grad_out"}},
                         ws, ws_bytes));
    const size_t need = ws_size("pairwise_softmax_matmul_backward", pr, C, 0);
    TP_CHECK(check_ws(ws, ws_bytes, need));
    TP_CHECK(injected_fault("pairwise_softmax_matmul_backward"));
    if (attn_tc_eligible(pr, sc, C, {V, out, lse, grad_out, dX, dY, dV})) {
        AttnTcArgs t{};
        t.Q = static_cast<const float*>(pr->X);
        t.K = static_cast<const float*>(pr->Y);
        t.V = static_cast<const float*>(V);
        t.N = pr->N;
        t.M = pr->M;
        t.scale = sc->scale;
        t.lse = static_cast<const float*>(lse);
        t.O = static_cast<const float*>(out);
        t.dO = static_cast<const float*>(grad_out);
        t.dQ = static_cast<float*>(dX);
        t.dK = static_cast<float*>(dY);
        t.dV = static_cast<float*>(dV);
        t.accumulate_dK = dX && dX == dY ? 1 : 0;  // same points: the column sweep adds dK onto dQ
        t.pm = (int)sc->pair_mask;
        t.band = pair_band(sc, pr);
        t.ws = ws;
        return tc_launched(launch_attn_bwd_tc(t, static_cast<cudaStream_t>(stream)));
    }
    // workspace: delta [N] first, partial states after it
    void* delta = ws;
    void* part = static_cast<char*>(ws) + align_up(pr->N * es);
    SweepArgs row = side_args(pr, sc, false), col = side_args(pr, sc, true);
    row.C = col.C = (int)C;
    row.Vp = grad_out;
    row.Vq = V;
    row.vecV = (cpad_bucket(row.C) == row.C && aligned(V, 16)) ? 1 : 0;
    col.Vp = V;
    col.Vq = grad_out;
    col.vecV = (cpad_bucket(col.C) == col.C && aligned(grad_out, 16)) ? 1 : 0;
    row.lse = col.lse = lse;
    row.delta = col.delta = delta;
    row.ws = col.ws = part;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return by_dtype(pr->dtype, [&](auto t) {
        using T = decltype(t);
        {
            HookScope h("softmax_delta", st);
            softmax_delta_kernel<T><<<(unsigned)cdiv(pr->N, 256), 256, 0, st>>>(
                static_cast<const T*>(grad_out), static_cast<const T*>(out), pr->N, (int)C, static_cast<T*>(delta));
        }
        return launched(1 + run_backward<T, kBSoftmax>(row, col, g, st));
    });
}

tp_status tp_pairwise_displacement_backward(const tp_pairs* pr, const tp_score* sc, const void* grad_out, void* dX,
                                            void* dY, void* d_row_bias, void* d_col_bias, void* d_row_weight,
                                            void* d_col_weight, void* ws, size_t ws_bytes, void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(grad_out, "grad_out", es));
    const Grads g{dX, dY, nullptr, d_row_bias, d_col_bias, d_row_weight, d_col_weight};
    TP_CHECK(check_grads(pr, sc, g, 1, {{grad_out, pr->N * pr->D * es, "grad_out"}}, ws, ws_bytes));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("pairwise_displacement_backward", pr, 0, 0)));
    TP_CHECK(injected_fault("pairwise_displacement_backward"));
    SweepArgs row = side_args(pr, sc, false), col = side_args(pr, sc, true);
    row.Vp = grad_out;
    col.Vq = grad_out;
    col.vecV = (pad_bucket(col.D) == col.D && aligned(grad_out, 16)) ? 1 : 0;
    row.ws = col.ws = ws;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return by_dtype(pr->dtype, [&](auto t) { return launched(run_backward<decltype(t), kBDisp>(row, col, g, st)); });
}

tp_status tp_pairwise_topk_backward(const tp_pairs* pr, const tp_score* sc, int k, const int64_t* indices,
                                    const void* grad_values, void* dX, void* dY, void* d_row_bias, void* d_col_bias,
                                    void* d_row_weight, void* d_col_weight, void* ws, size_t ws_bytes,
                                    void* stream) {
    TP_CHECK(check_pairs(pr));
    TP_CHECK(check_score(sc, pr));
    if (k < 1 || k > pr->M || k > 128) return fail(TP_ERR_INVALID_ARG, "k must be in [1, min(M, 128)]");
    if (pr->N * (int64_t)k >= (int64_t(1) << 31)) return fail(TP_ERR_INVALID_ARG, "N * k must be below 2^31");
    const size_t es = esize(pr->dtype);
    TP_CHECK(check_ptr(indices, "indices", 8));
    TP_CHECK(check_ptr(grad_values, "grad_values", es));
    const Grads g{dX, dY, nullptr, d_row_bias, d_col_bias, d_row_weight, d_col_weight};
    TP_CHECK(check_grads(pr, sc, g, 1,
                         {{indices, (size_t)(pr->N * k) * 8, "indices"}, {grad_values, (size_t)(pr->N * k) * es, "grad_values"}}, ws,
                         ws_bytes));
    TP_CHECK(check_ws(ws, ws_bytes, ws_size("pairwise_topk_backward", pr, 0, k)));
    TP_CHECK(injected_fault("pairwise_topk_backward"));
    SweepArgs row = side_args(pr, sc, false), col = side_args(pr, sc, true);
    row.k = col.k = k;
    row.gP = dX;
    row.gPb = d_row_bias;
    row.gPw = d_row_weight;
    col.gP = dY;
    col.gPb = d_col_bias;
    col.gPw = d_col_weight;
    col.accumulate = (dY && dY == dX) ? 1 : 0;
    char* w = static_cast<char*>(ws);
    const size_t mb = align_up(pr->M * 4);
    int* count = reinterpret_cast<int*>(w);
    int* cursor = reinterpret_cast<int*>(w + mb);
    int* bucket = reinterpret_cast<int*>(w + 2 * mb);
    int* start = reinterpret_cast<int*>(w + 2 * mb + align_up((size_t)pr->N * k * 4));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool cols = dY || d_col_bias || d_col_weight;
    if (cols && cudaMemsetAsync(count, 0, pr->M * 4, st) != cudaSuccess) return launched(0);
    return by_dtype(pr->dtype, [&](auto t) {
        using T = decltype(t);
        launch_topk_bwd<T>(row, col, indices, grad_values, count, start, cursor, bucket, st);
        const bool rows = dX || d_row_bias || d_row_weight;
        return launched((rows ? 1 : 0) + (cols ? 4 : 0));
    });
}

}  // extern "C"
