// Generic SIMT sweep kernels for every consumer (fp32 and fp64, any D and C up to 64).
//
// Layout of one launch: grid = (ceil(nP / 128), splits). A CTA owns 128 consecutive points of the
// "own" set P (one per thread, held in registers) and streams the points of the other set Q in
// [begin, end) of its split through shared memory, 32 at a time; every thread reads the staged row
// with 16-byte broadcast loads. Forward: P = X (rows), Q = Y. Backward row sweep: the same.
// Backward column sweep: P = Y, Q = X with row/column parameters swapped, which is the transposed
// sweep that lets every output be owned by exactly one thread, so no atomics are needed.
// With splits > 1 each CTA writes its partial state to the caller's workspace ([split][w][nP]) and a
// merge kernel combines the splits in fixed order: results are deterministic.
//
// Method: torchpairwise guide "Using Torchpairwise in Models" (introduction: consume in bounded
// tiles, never store [N,M], replay tiles for first derivatives; "Task Map": softmax_matmul, K @ V,
// logsumexp with exclude_self, topk with exact tie order; "Stein Variational Gradient Descent":
// displacement and the SVGD direction).
#pragma once

#include <type_traits>

#include "tp_args.h"
#include "tp_device.cuh"
#include "tp_launch.h"

namespace tp {

// Whether the pair of own point pi and streamed point qj stays in the consumer's reduction under the
// sweep's pair mask (torchpairwise guide "Using Torchpairwise in Models", Score Expressions: tp.masks
// causal, band, same_group). og: the own point's group id (same-group masks only).
__device__ __forceinline__ bool pair_kept(const SweepArgs& a, int64_t pi, int64_t qj, int og) {
    const int64_t i = a.pcol ? qj : pi, j = a.pcol ? pi : qj;
    switch (a.pm) {
        case 1: return j <= i;
        case 2: return (i > j ? i - j : j - i) <= a.band;
        case 3: return __ldg(a.qg + qj) == og;
        default: return true;
    }
}

// ------------------------------------------------------------------------------------------------
// two-level accumulation
// ------------------------------------------------------------------------------------------------
//
// Every sum over the streamed set is kept in two levels: a register accumulator for the current
// 32-point tile and a running accumulator that the tile's sum is added into once per tile. The
// rounding of one sum then grows with 32 + n/32 instead of n. Vector running accumulators live in
// shared memory, column-major ([width][kThreads]) so that each thread touches its own bank.

template <class T>
__host__ __device__ constexpr size_t al16(size_t nelem) {
    return (nelem * sizeof(T) + 15) / 16 * 16;
}

template <class T, int N>
struct RunningVec {
    T* base;  // [N][kThreads] in shared memory
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int c = 0; c < N; ++c) base[c * kThreads + threadIdx.x] = T(0);
    }
    // running = running * r + tile; tile = 0
    __device__ __forceinline__ void flush(T (&tile)[N], T r) {
#pragma unroll
        for (int c = 0; c < N; ++c) {
            T& v = base[c * kThreads + threadIdx.x];
            v = fma(v, r, tile[c]);
            tile[c] = T(0);
        }
    }
    __device__ __forceinline__ void flush(T (&tile)[N]) {
#pragma unroll
        for (int c = 0; c < N; ++c) {
            base[c * kThreads + threadIdx.x] += tile[c];
            tile[c] = T(0);
        }
    }
    __device__ __forceinline__ T get(int c) const { return base[c * kThreads + threadIdx.x]; }
};

template <class T>
struct Running {
    T run = T(0), tile = T(0);
    __device__ __forceinline__ void flush() {
        run += tile;
        tile = T(0);
    }
    __device__ __forceinline__ void flush(T r) {
        run = fma(run, r, tile);
        tile = T(0);
    }
};

// Dynamic shared memory of the forward sweep, carved in this order: staged points [kTile][DP],
// staged values [kTile][VW], norms, column weights, column biases, running accumulators.
template <class T, int DP, int CP, int MODE, bool AFFINE>
struct FwdSmem {
    static constexpr bool HAS_V = MODE == kMatmul || MODE == kSoftmax || MODE == kSvgd;
    static constexpr int VW = MODE == kSvgd ? DP : CP;
    static constexpr int NRUN = (MODE == kMatmul || MODE == kSoftmax) ? CP : (MODE == kDisp || MODE == kSvgd ? DP : 0);
    static constexpr size_t bytes = al16<T>(kTile * DP) + (HAS_V ? al16<T>(kTile * VW) : 0) + al16<T>(kTile) +
                                    (AFFINE ? 2 * al16<T>(kTile) : 0) + al16<T>((size_t)NRUN * kThreads);
};

// Dynamic shared memory of a backward sweep: staged points, staged values, norms, weights, biases,
// two per-row statistics, running accumulators ([K1 | Kd | dV]).
template <class T, int DP, int CP, int MODE, int SIDE, bool DO_G, bool DO_V>
struct BwdSmem {
    static constexpr bool VALS = MODE == kBMatmul || MODE == kBSoftmax;
    static constexpr int QVW = VALS ? CP : ((MODE == kBDisp && SIDE == kCol) ? DP : 1);
    static constexpr bool HAS_QV = VALS || (MODE == kBDisp && SIDE == kCol);
    static constexpr int NK1 = DO_G ? DP : 0;
    static constexpr int NKD = (DO_G && MODE == kBDisp && SIDE == kCol) ? DP : 0;
    static constexpr int NKV = DO_V ? CP : 0;
    static constexpr size_t bytes = al16<T>(kTile * DP) + (HAS_QV ? al16<T>(kTile * QVW) : 0) + 5 * al16<T>(kTile) +
                                    al16<T>((size_t)(NK1 + NKD + NKV) * kThreads);
};

struct SmemCursor {
    unsigned char* p;
    template <class T>
    __device__ __forceinline__ T* take(size_t nelem) {
        T* r = reinterpret_cast<T*>(p);
        p += al16<T>(nelem);
        return r;
    }
};

// ------------------------------------------------------------------------------------------------
// forward sweep
// ------------------------------------------------------------------------------------------------

template <int MODE>
__host__ __device__ inline int fwd_state_width(int D, int C) {
    return MODE == kMatmul ? C : MODE == kSoftmax ? 2 + C : MODE == kLse ? 2 : D + 1;  // kDisp, kSvgd: D sums + mass
}

template <class T, int DP, int CP, int MODE, bool AFFINE>
__global__ void __launch_bounds__(kThreads) fwd_sweep(const SweepArgs a) {
    griddep_wait();  // launched with launch_pdl: nothing before this touches global memory
    using E = ExpTraits<T>;
    using SM = FwdSmem<T, DP, CP, MODE, AFFINE>;
    constexpr bool HAS_V = SM::HAS_V;
    constexpr int VW = SM::VW;
    constexpr int NACC = (MODE == kMatmul || MODE == kSoftmax) ? CP : (MODE == kLse ? 1 : DP);
    constexpr bool VEC_RUN = SM::NRUN > 0;

    extern __shared__ __align__(16) unsigned char tp_smem[];
    SmemCursor cur{tp_smem};
    T* sq = cur.take<T>(kTile * DP);
    T* sv = HAS_V ? cur.take<T>(kTile * VW) : nullptr;
    T* sn = cur.take<T>(kTile);
    T* sw = AFFINE ? cur.take<T>(kTile) : nullptr;
    T* sb = AFFINE ? cur.take<T>(kTile) : nullptr;
    RunningVec<T, NACC> run1{cur.take<T>((size_t)SM::NRUN * kThreads)};

    const T* __restrict__ P = static_cast<const T*>(a.P);
    const T* __restrict__ Q = static_cast<const T*>(a.Q);
    const int64_t pi = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const bool pvalid = pi < a.nP;
    const int split = blockIdx.y;
    const int64_t jb = (int64_t)split * a.cps;
    const int64_t je = min(a.nQ, jb + a.cps);

    T p[DP];
    load_point<T, DP>(p, P, pi, a.D, pvalid);
    const T pn = a.metric != kLinear ? sqnorm<T, DP>(p) : T(0);
    const T neg_gamma = T(-a.gamma);
    T A = T(a.scale), Cp = T(0);
    if constexpr (AFFINE) {
        if (pvalid && a.pw) A *= static_cast<const T*>(a.pw)[pi];
        if (pvalid && a.pb) Cp = static_cast<const T*>(a.pb)[pi];
    }
    const int og = (a.pm == 3 && pvalid) ? a.pg[pi] : 0;

    // tile accumulators (registers); running accumulators (shared memory / scalars)
    T acc[NACC];
#pragma unroll
    for (int c = 0; c < NACC; ++c) acc[c] = T(0);
    if constexpr (VEC_RUN) {
        run1.init();
    }
    T m = ninf<T>();
    Running<T> l, mass;

    zero_smem(sq, kTile * DP);
    if constexpr (HAS_V) zero_smem(sv, kTile * VW);

    // the tile loop, compiled once without and once with the pair mask test (chosen per launch)
    auto sweep = [&](auto masked) {
        for (int64_t j0 = jb; j0 < je; j0 += kTile) {
            const int cnt = (int)(je - j0 < (int64_t)kTile ? je - j0 : (int64_t)kTile);
            __syncthreads();
            stage_rows<T, DP>(sq, Q, j0, cnt, a.D, a.vecQ);
            if constexpr (HAS_V)
                stage_rows<T, VW>(sv, static_cast<const T*>(a.Vq), j0, cnt, MODE == kSvgd ? a.D : a.C, a.vecV);
            if constexpr (AFFINE) {
                stage_scalar<T>(sw, static_cast<const T*>(a.qw), j0, cnt, T(1));
                stage_scalar<T>(sb, static_cast<const T*>(a.qb), j0, cnt, T(0));
            }
            __syncthreads();
            if (a.metric != kLinear) {
                stage_norms<T, DP>(sn, sq, cnt);
                if constexpr (MODE == kSvgd) {  // the staged values become w_j = score_j - 2 gamma x_j
                    const T g2 = T(2 * a.gamma);
                    for (int e = threadIdx.x; e < cnt * DP; e += kThreads) sv[e] = fma(-g2, sq[e], sv[e]);
                }
                __syncthreads();
            }
            const T m0 = m;  // the running state is relative to the max at the start of the tile
    #pragma unroll 2
            for (int jj = 0; jj < cnt; ++jj) {
                if constexpr (decltype(masked)::value)
                    if (!pair_kept(a, pi, j0 + jj, og)) continue;  // a masked pair adds nothing
                const T* q = sq + jj * DP;
                const T base = pair_base<T, DP>(a.metric, p, q, pn, sn[jj], neg_gamma);
                T t;
                if constexpr (AFFINE) t = fma(A * sw[jj], base, Cp + sb[jj]);
                else t = A * base;
                const T S = a.apply_exp ? E::exp(t) : t;
                if constexpr (MODE == kMatmul) {
                    axpy_smem<T, CP>(acc, S, sv + jj * CP);
                } else if constexpr (MODE == kLse || MODE == kSoftmax) {
                    if (MODE == kLse && a.exclude_self && j0 + jj == pi) continue;
                    const T s = S * E::kLogB;
                    if (s > m) {
                        const T r = E::bexp(m - s);
                        l.tile *= r;
                        if constexpr (MODE == kSoftmax) {
    #pragma unroll
                            for (int c = 0; c < CP; ++c) acc[c] *= r;
                        }
                        m = s;
                    }
                    const T pr = s > ninf<T>() ? E::bexp(s - m) : T(0);  // an empty element (-inf) adds 0, not NaN
                    l.tile += pr;
                    if constexpr (MODE == kSoftmax) axpy_smem<T, CP>(acc, pr, sv + jj * CP);
                } else if constexpr (MODE == kDisp) {
                    axpy_smem<T, DP>(acc, S, q);
                    mass.tile += S;
                } else {  // kSvgd: S is the bare rbf kernel value k_ij; the staged row is w_j = score_j - 2 gamma x_j
                    axpy_smem<T, DP>(acc, S, sv + jj * DP);
                    mass.tile += S;
                }
            }
            if constexpr (MODE == kLse || MODE == kSoftmax) {
                // 0 while the running state is empty (m0 = -inf); 1 when the max did not move (this also
                // covers a tile with no admitted pair, where both are -inf)
                const T r = m0 == m ? T(1) : E::bexp(m0 - m);
                l.flush(r);
                if constexpr (MODE == kSoftmax) run1.flush(acc, r);
            } else {
                if constexpr (VEC_RUN) run1.flush(acc);
                mass.flush();
            }
        }
    };
    if (a.pm) sweep(std::true_type{});
    else sweep(std::false_type{});
    if (!pvalid) return;
    const T L = l.run, MASS = mass.run;

    if (a.splits > 1) {
        T* ws = static_cast<T*>(a.ws);
        const int W = fwd_state_width<MODE>(a.D, a.C);
        T* o = ws + (int64_t)split * W * a.nP + pi;
        if constexpr (MODE == kMatmul) {
#pragma unroll
            for (int c = 0; c < CP; ++c)
                if (c < a.C) o[(int64_t)c * a.nP] = run1.get(c);
        } else if constexpr (MODE == kSoftmax) {
            o[0] = m;
            o[a.nP] = L;
#pragma unroll
            for (int c = 0; c < CP; ++c)
                if (c < a.C) o[(int64_t)(2 + c) * a.nP] = run1.get(c);
        } else if constexpr (MODE == kLse) {
            o[0] = m;
            o[a.nP] = L;
        } else if constexpr (MODE == kDisp) {
#pragma unroll
            for (int d = 0; d < DP; ++d)
                if (d < a.D) o[(int64_t)d * a.nP] = run1.get(d);
            o[(int64_t)a.D * a.nP] = MASS;
        } else {
#pragma unroll
            for (int d = 0; d < DP; ++d)
                if (d < a.D) o[(int64_t)d * a.nP] = run1.get(d);
            o[(int64_t)a.D * a.nP] = MASS;
        }
        return;
    }

    T* out = static_cast<T*>(a.out);
    if constexpr (MODE == kMatmul) {
#pragma unroll
        for (int c = 0; c < CP; ++c)
            if (c < a.C) out[pi * a.C + c] = run1.get(c);
    } else if constexpr (MODE == kSoftmax) {
        const T inv = L > T(0) ? T(1) / L : T(0);  // a row with every pair masked returns 0
#pragma unroll
        for (int c = 0; c < CP; ++c)
            if (c < a.C) out[pi * a.C + c] = run1.get(c) * inv;
        static_cast<T*>(a.out2)[pi] = E::lse(m, L);
    } else if constexpr (MODE == kLse) {
        out[pi] = L > T(0) ? E::lse(m, L) : ninf<T>();
    } else if constexpr (MODE == kDisp) {
#pragma unroll
        for (int d = 0; d < DP; ++d)
            if (d < a.D) out[pi * a.D + d] = run1.get(d) - MASS * p[d];
    } else {
        // phi_i = (sum_j k_ij (score_j - 2 gamma x_j) + 2 gamma x_i sum_j k_ij) / n
        const T g2 = T(2 * a.gamma), inv_n = T(a.inv_n);
#pragma unroll
        for (int d = 0; d < DP; ++d)
            if (d < a.D) out[pi * a.D + d] = fma(g2 * MASS, p[d], run1.get(d)) * inv_n;
    }
}

// Combine the per-split partial states of a forward sweep, splits in ascending order.
template <class T, int MODE>
__global__ void __launch_bounds__(kThreads) fwd_merge(const SweepArgs a) {
    griddep_wait();  // launched with launch_pdl: nothing before this touches global memory
    using E = ExpTraits<T>;
    const int64_t pi = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (pi >= a.nP) return;
    const T* ws = static_cast<const T*>(a.ws);
    const int W = fwd_state_width<MODE>(a.D, a.C);
    const int64_t sstride = (int64_t)W * a.nP;
    T* out = static_cast<T*>(a.out);
    if constexpr (MODE == kMatmul) {
        for (int c = 0; c < a.C; ++c) {
            T s = T(0);
            for (int sp = 0; sp < a.splits; ++sp) s += ws[sp * sstride + (int64_t)c * a.nP + pi];
            out[pi * a.C + c] = s;
        }
    } else if constexpr (MODE == kSoftmax || MODE == kLse) {
        T m = ninf<T>();
        for (int sp = 0; sp < a.splits; ++sp) m = fmax(m, ws[sp * sstride + pi]);
        T l = T(0);
        for (int sp = 0; sp < a.splits; ++sp) {
            const T ms = ws[sp * sstride + pi];
            if (ms > ninf<T>()) l += ws[sp * sstride + a.nP + pi] * E::bexp(ms - m);
        }
        const T lse = l > T(0) ? E::lse(m, l) : ninf<T>();
        if constexpr (MODE == kLse) {
            out[pi] = lse;
        } else {
            static_cast<T*>(a.out2)[pi] = lse;
            const T inv = l > T(0) ? T(1) / l : T(0);  // a row with every pair masked returns 0
            for (int c = 0; c < a.C; ++c) {
                T s = T(0);
                for (int sp = 0; sp < a.splits; ++sp) {
                    const T ms = ws[sp * sstride + pi];
                    if (ms > ninf<T>()) s += ws[sp * sstride + (int64_t)(2 + c) * a.nP + pi] * E::bexp(ms - m);
                }
                out[pi * a.C + c] = s * inv;
            }
        }
    } else {
        const T* P = static_cast<const T*>(a.P);
        T mass = T(0);
        for (int sp = 0; sp < a.splits; ++sp) mass += ws[sp * sstride + (int64_t)a.D * a.nP + pi];
        for (int d = 0; d < a.D; ++d) {
            T s1 = T(0);
            for (int sp = 0; sp < a.splits; ++sp) s1 += ws[sp * sstride + (int64_t)d * a.nP + pi];
            const T pd = P[pi * a.D + d];
            if (MODE == kDisp) out[pi * a.D + d] = s1 - mass * pd;
            else out[pi * a.D + d] = fma(T(2 * a.gamma) * mass, pd, s1) * T(a.inv_n);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// top-k (k smallest keys; key = S, or -S for largest), exact (value, index) order
// ------------------------------------------------------------------------------------------------

constexpr int kNoIndex = 0x7fffffff;

template <class T, int DP, int K, bool AFFINE>
__global__ void __launch_bounds__(kThreads) topk_sweep(const SweepArgs a) {
    griddep_wait();  // launched with launch_pdl: nothing before this touches global memory
    using E = ExpTraits<T>;
    __shared__ __align__(16) T sq[kTile * DP];
    __shared__ T sn[kTile];
    __shared__ T sw[AFFINE ? kTile : 1];
    __shared__ T sb[AFFINE ? kTile : 1];

    const T* __restrict__ P = static_cast<const T*>(a.P);
    const T* __restrict__ Q = static_cast<const T*>(a.Q);
    const int64_t pi = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const bool pvalid = pi < a.nP;
    const int split = blockIdx.y;
    const int64_t jb = (int64_t)split * a.cps;
    const int64_t je = min(a.nQ, jb + a.cps);

    T p[DP];
    load_point<T, DP>(p, P, pi, a.D, pvalid);
    const T pn = a.metric != kLinear ? sqnorm<T, DP>(p) : T(0);
    const T neg_gamma = T(-a.gamma);
    T A = T(a.scale), Cp = T(0);
    if constexpr (AFFINE) {
        if (pvalid && a.pw) A *= static_cast<const T*>(a.pw)[pi];
        if (pvalid && a.pb) Cp = static_cast<const T*>(a.pb)[pi];
    }
    const T sgn = a.largest ? T(-1) : T(1);
    const int og = (a.pm == 3 && pvalid) ? a.pg[pi] : 0;

    T kv[K];
    int ki[K];
#pragma unroll
    for (int t = 0; t < K; ++t) {
        kv[t] = pinf<T>();
        ki[t] = kNoIndex;
    }
    zero_smem(sq, kTile * DP);
    // the tile loop, compiled once without and once with the pair mask test (chosen per launch)
    auto sweep = [&](auto masked) {
        for (int64_t j0 = jb; j0 < je; j0 += kTile) {
            const int cnt = (int)(je - j0 < (int64_t)kTile ? je - j0 : (int64_t)kTile);
            __syncthreads();
            stage_rows<T, DP>(sq, Q, j0, cnt, a.D, a.vecQ);
            if constexpr (AFFINE) {
                stage_scalar<T>(sw, static_cast<const T*>(a.qw), j0, cnt, T(1));
                stage_scalar<T>(sb, static_cast<const T*>(a.qb), j0, cnt, T(0));
            }
            __syncthreads();
            if (a.metric != kLinear) {
                stage_norms<T, DP>(sn, sq, cnt);
                __syncthreads();
            }
    #pragma unroll 4
            for (int jj = 0; jj < cnt; ++jj) {
                if constexpr (decltype(masked)::value)
                    if (!pair_kept(a, pi, j0 + jj, og)) continue;  // a masked pair is never selected
                const T base = pair_base<T, DP>(a.metric, p, sq + jj * DP, pn, sn[jj], neg_gamma);
                T t;
                if constexpr (AFFINE) t = fma(A * sw[jj], base, Cp + sb[jj]);
                else t = A * base;
                const T S = a.apply_exp ? E::exp(t) : t;
                topk_insert<T, K>(kv, ki, sgn * S, (int)(j0 + jj));
            }
        }
    };
    if (a.pm) sweep(std::true_type{});
    else sweep(std::false_type{});
    if (!pvalid) return;
    if (a.splits > 1) {
        T* wv = static_cast<T*>(a.ws);
        int* wi = reinterpret_cast<int*>(wv + (int64_t)a.splits * K * a.nP);
#pragma unroll
        for (int t = 0; t < K; ++t) {
            if (t < a.k) {
                const int64_t o = ((int64_t)split * K + t) * a.nP + pi;
                wv[o] = kv[t];
                wi[o] = ki[t];
            }
        }
        return;
    }
    T* vals = static_cast<T*>(a.out);
    int64_t* idx = static_cast<int64_t*>(a.out2);
#pragma unroll
    for (int t = 0; t < K; ++t)
        if (t < a.k) {
            vals[pi * a.k + t] = sgn * kv[t];
            idx[pi * a.k + t] = ki[t] == kNoIndex ? -1 : ki[t];  // fewer than k kept pairs: (+-inf, -1)
        }
}

template <class T, int K>
__global__ void __launch_bounds__(kThreads) topk_merge(const SweepArgs a) {
    griddep_wait();  // launched with launch_pdl: nothing before this touches global memory
    const int64_t pi = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (pi >= a.nP) return;
    const T* wv = static_cast<const T*>(a.ws);
    const int* wi = reinterpret_cast<const int*>(wv + (int64_t)a.splits * K * a.nP);
    T kv[K];
    int ki[K];
#pragma unroll
    for (int t = 0; t < K; ++t) {
        kv[t] = pinf<T>();
        ki[t] = kNoIndex;
    }
    for (int sp = 0; sp < a.splits; ++sp)
        for (int t = 0; t < a.k; ++t) {
            const int64_t o = ((int64_t)sp * K + t) * a.nP + pi;
            topk_insert_lex<T, K>(kv, ki, wv[o], wi[o]);
        }
    const T sgn = a.largest ? T(-1) : T(1);
    T* vals = static_cast<T*>(a.out);
    int64_t* idx = static_cast<int64_t*>(a.out2);
#pragma unroll
    for (int t = 0; t < K; ++t)
        if (t < a.k) {
            vals[pi * a.k + t] = sgn * kv[t];
            idx[pi * a.k + t] = ki[t] == kNoIndex ? -1 : ki[t];  // fewer than k kept pairs: (+-inf, -1)
        }
}

// ------------------------------------------------------------------------------------------------
// backward replay sweeps
// ------------------------------------------------------------------------------------------------
//
// For an upstream G_pq = dL/dS_pq, H = dL/dt = G (times S when exp is applied), E = dL/dbase =
// H * scale * w_p * w_q, and the own point's gradient is sum_q kappa q - [distance metric] p sum_q kappa
// with kappa = E (linear), -2E (sqeuclidean), 2 gamma E base (rbf). Own bias gradient = sum_q H,
// own weight gradient = sum_q H scale w_q base.
// G per consumer (row sweep p = x_i, q = y_j; column sweep p = y_j, q = x_i):
//   matmul  : dO_i . V_j                   ; dV_j = sum_i S_ij dO_i
//   softmax : P_ij (dO_i . V_j - delta_i)  ; dV_j = sum_i P_ij dO_i ; P_ij = exp(S_ij - lse_i)
//   lse     : g_i P_ij (0 for the excluded pair)
//   disp    : dO_i . (y_j - x_i), plus the direct terms -dO_i sum_j S_ij (dX) and sum_i S_ij dO_i (dY).

// partial-state width of a backward sweep: [K1 (D), K0, sumH, sumHw, extra...]
template <int MODE, int SIDE, bool DO_G, bool DO_V>
__host__ __device__ inline int bwd_state_width(int D, int C) {
    int w = 0;
    if (DO_G) {
        w += D + 3;
        if (MODE == kBDisp) w += SIDE == kRow ? 1 : D;
    }
    if (DO_V) w += C;
    return w;
}

template <class T, int DP, int CP, int MODE, int SIDE, bool DO_G, bool DO_V>
__global__ void __launch_bounds__(kThreads) bwd_sweep(const SweepArgs a) {
    griddep_wait();  // launched with launch_pdl: nothing before this touches global memory
    using E = ExpTraits<T>;
    constexpr bool VALS = MODE == kBMatmul || MODE == kBSoftmax;
    // own value vector: row sweep dO_i (CP; DP for disp); column sweep V_j (CP) when DO_G
    constexpr int PVW = (MODE == kBDisp && SIDE == kRow) ? DP : ((VALS && (SIDE == kRow || DO_G)) ? CP : 1);
    // staged value rows: row sweep V_j (CP); column sweep dO_i (CP; DP for disp)
    constexpr int QVW = VALS ? CP : ((MODE == kBDisp && SIDE == kCol) ? DP : 1);
    constexpr bool HAS_QV = VALS || (MODE == kBDisp && SIDE == kCol);
    constexpr bool ROWSTAT = (MODE == kBSoftmax || MODE == kBLse || MODE == kBLseSym);
    constexpr bool QSTAT = (SIDE == kCol && ROWSTAT) || MODE == kBLseSym;  // per-streamed-point lse, g
    constexpr int KD = (MODE == kBDisp && SIDE == kCol) ? DP : 1;

    using SM = BwdSmem<T, DP, CP, MODE, SIDE, DO_G, DO_V>;
    extern __shared__ __align__(16) unsigned char tp_smem[];
    SmemCursor cur{tp_smem};
    T* sq = cur.take<T>(kTile * DP);
    T* sv = HAS_QV ? cur.take<T>(kTile * QVW) : nullptr;
    T* sn = cur.take<T>(kTile);
    T* sw = cur.take<T>(kTile);
    T* sb = cur.take<T>(kTile);
    T* s1 = cur.take<T>(kTile);  // column sweep: lse_i (base domain) / dO_i . x_i (disp)
    T* s2 = cur.take<T>(kTile);  // column sweep: delta_i (softmax) / g_i (lse)
    T* runbase = cur.take<T>((size_t)(SM::NK1 + SM::NKD + SM::NKV) * kThreads);
    RunningVec<T, DO_G ? DP : 1> rK1{runbase};
    RunningVec<T, KD> rKd{runbase + (size_t)SM::NK1 * kThreads};
    RunningVec<T, DO_V ? CP : 1> rKV{runbase + (size_t)(SM::NK1 + SM::NKD) * kThreads};

    const T* __restrict__ P = static_cast<const T*>(a.P);
    const T* __restrict__ Q = static_cast<const T*>(a.Q);
    const int64_t pi = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const bool pvalid = pi < a.nP;
    const int split = blockIdx.y;
    const int64_t jb = (int64_t)split * a.cps;
    const int64_t je = min(a.nQ, jb + a.cps);

    T p[DP];
    load_point<T, DP>(p, P, pi, a.D, pvalid);
    const T pn = a.metric != kLinear ? sqnorm<T, DP>(p) : T(0);
    const T neg_gamma = T(-a.gamma);
    const T scale = T(a.scale);
    T wp = T(1), bp = T(0);
    if (pvalid && a.pw) wp = static_cast<const T*>(a.pw)[pi];
    if (pvalid && a.pb) bp = static_cast<const T*>(a.pb)[pi];
    const int og = (a.pm == 3 && pvalid) ? a.pg[pi] : 0;
    const T A = scale * wp;
    const bool affine = a.affine != 0;

    // own value vector and per-row statistics
    T pv[PVW];
#pragma unroll
    for (int c = 0; c < PVW; ++c) pv[c] = T(0);
    T plse = T(0), pstat = T(0);  // row sweep: lse_i (base domain), delta_i / g_i / dO_i.x_i
    if (pvalid) {
        if constexpr (PVW > 1) {
            const int W = (MODE == kBDisp) ? a.D : a.C;
            const T* vp = static_cast<const T*>(a.Vp) + pi * W;
#pragma unroll
            for (int c = 0; c < PVW; ++c)
                if (c < W) pv[c] = vp[c];
        }
        if constexpr (SIDE == kRow) {
            if constexpr (ROWSTAT) plse = static_cast<const T*>(a.lse)[pi] * E::kLogB;
            if constexpr (MODE == kBSoftmax) pstat = static_cast<const T*>(a.delta)[pi];
            if constexpr (MODE == kBLse || MODE == kBLseSym) pstat = static_cast<const T*>(a.glse)[pi];
            if constexpr (MODE == kBDisp) {
                T c0 = T(0);
#pragma unroll
                for (int d = 0; d < DP; ++d) c0 = fma(pv[d], p[d], c0);
                pstat = c0;
            }
        }
    }

    T K1[DO_G ? DP : 1];
    T KdV[DO_V ? CP : 1];
    T Kd[KD];
#pragma unroll
    for (int d = 0; d < (DO_G ? DP : 1); ++d) K1[d] = T(0);
#pragma unroll
    for (int c = 0; c < (DO_V ? CP : 1); ++c) KdV[c] = T(0);
#pragma unroll
    for (int d = 0; d < KD; ++d) Kd[d] = T(0);
    Running<T> K0, sumH, sumHw, sumS;
    if constexpr (DO_G) rK1.init();
    if constexpr (SM::NKD > 0) rKd.init();
    if constexpr (DO_V) rKV.init();

    zero_smem(sq, kTile * DP);
    if constexpr (HAS_QV) zero_smem(sv, kTile * QVW);

    // the tile loop, compiled once without and once with the pair mask test (chosen per launch)
    auto sweep = [&](auto masked) {
        for (int64_t j0 = jb; j0 < je; j0 += kTile) {
            const int cnt = (int)(je - j0 < (int64_t)kTile ? je - j0 : (int64_t)kTile);
            __syncthreads();
            stage_rows<T, DP>(sq, Q, j0, cnt, a.D, a.vecQ);
            if constexpr (HAS_QV)
                stage_rows<T, QVW>(sv, static_cast<const T*>(a.Vq), j0, cnt, MODE == kBDisp ? a.D : a.C, a.vecV);
            stage_scalar<T>(sw, static_cast<const T*>(a.qw), j0, cnt, T(1));
            stage_scalar<T>(sb, static_cast<const T*>(a.qb), j0, cnt, T(0));
            if constexpr (QSTAT) {
                for (int e = threadIdx.x; e < cnt; e += kThreads) {
                    s1[e] = static_cast<const T*>(a.lse)[j0 + e] * E::kLogB;
                    s2[e] = MODE == kBSoftmax ? static_cast<const T*>(a.delta)[j0 + e]
                                              : static_cast<const T*>(a.glse)[j0 + e];
                }
            }
            __syncthreads();
            if (a.metric != kLinear) stage_norms<T, DP>(sn, sq, cnt);
            if constexpr (SIDE == kCol && MODE == kBDisp) {
                for (int r = threadIdx.x; r < cnt; r += kThreads) {
                    T c0 = T(0);
                    for (int d = 0; d < DP; ++d) c0 = fma(sv[r * QVW + d], sq[r * DP + d], c0);
                    s1[r] = c0;
                }
            }
            __syncthreads();
    #pragma unroll 2
            for (int jj = 0; jj < cnt; ++jj) {
                if constexpr (decltype(masked)::value)
                    if (!pair_kept(a, pi, j0 + jj, og)) continue;  // a masked pair has no gradient
                const T* q = sq + jj * DP;
                const T base = pair_base<T, DP>(a.metric, p, q, pn, sn[jj], neg_gamma);
                const T wq = sw[jj];
                const T t = affine ? fma(A * wq, base, bp + sb[jj]) : A * base;
                const T S = a.apply_exp ? E::exp(t) : t;
                T G = T(0), Pw = S;
                if constexpr (MODE == kBMatmul) {
                    if constexpr (DO_G) G = dot_regs_smem<T, CP>(pv, sv + jj * CP);
                } else if constexpr (MODE == kBSoftmax) {
                    const T lse_b = SIDE == kRow ? plse : s1[jj];
                    Pw = E::bexp(S * E::kLogB - lse_b);
                    if constexpr (DO_G) {
                        const T dl = SIDE == kRow ? pstat : s2[jj];
                        G = Pw * (dot_regs_smem<T, CP>(pv, sv + jj * CP) - dl);
                    }
                } else if constexpr (MODE == kBLse) {
                    const T lse_b = SIDE == kRow ? plse : s1[jj];
                    const T g = SIDE == kRow ? pstat : s2[jj];
                    const bool excluded = a.exclude_self && (j0 + jj == pi);
                    G = (excluded || !(lse_b > ninf<T>())) ? T(0) : g * E::bexp(S * E::kLogB - lse_b);
                } else if constexpr (MODE == kBLseSym) {
                    // the pair seen from row k (this thread) and from row j (the streamed point)
                    const bool excluded = a.exclude_self && (j0 + jj == pi);
                    const T sb2 = S * E::kLogB;
                    const T gk = plse > ninf<T>() ? pstat * E::bexp(sb2 - plse) : T(0);
                    const T gj = s1[jj] > ninf<T>() ? s2[jj] * E::bexp(sb2 - s1[jj]) : T(0);
                    G = excluded ? T(0) : gk + gj;
                } else {  // kBDisp
                    if constexpr (SIDE == kRow) {
                        G = dot_regs_smem<T, DP>(pv, q) - pstat;
                        sumS.tile += S;
                    } else {
                        const T* dO = sv + jj * DP;
                        G = dot_regs_smem<T, DP>(p, dO) - s1[jj];
                        axpy_smem<T, DP>(Kd, S, dO);
                    }
                }
                if constexpr (DO_V) axpy_smem<T, CP>(KdV, Pw, sv + jj * CP);
                if constexpr (DO_G) {
                    const T H = a.apply_exp ? G * S : G;
                    sumH.tile += H;
                    if (affine) sumHw.tile = fma(H * scale * wq, base, sumHw.tile);
                    const T Ev = H * A * wq;
                    const T kappa = a.metric == kLinear ? Ev : (a.metric == kSqeuclidean ? T(-2) * Ev : T(-2) * neg_gamma * Ev * base);
                    K0.tile += kappa;
                    axpy_smem<T, DP>(K1, kappa, q);
                }
            }
            if constexpr (DO_G) {
                rK1.flush(K1);
                K0.flush();
                sumH.flush();
                sumHw.flush();
                sumS.flush();
            }
            if constexpr (SM::NKD > 0) rKd.flush(Kd);
            if constexpr (DO_V) rKV.flush(KdV);
        }
    };
    if (a.pm) sweep(std::true_type{});
    else sweep(std::false_type{});
    if (!pvalid) return;

    if (a.splits > 1) {
        T* ws = static_cast<T*>(a.ws);
        const int W = bwd_state_width<MODE, SIDE, DO_G, DO_V>(a.D, a.C);
        T* o = ws + (int64_t)split * W * a.nP + pi;
        int w = 0;
        if constexpr (DO_G) {
#pragma unroll
            for (int d = 0; d < DP; ++d)
                if (d < a.D) o[(int64_t)(w + d) * a.nP] = rK1.get(d);
            w += a.D;
            o[(int64_t)w++ * a.nP] = K0.run;
            o[(int64_t)w++ * a.nP] = sumH.run;
            o[(int64_t)w++ * a.nP] = sumHw.run;
            if constexpr (MODE == kBDisp && SIDE == kRow) o[(int64_t)w++ * a.nP] = sumS.run;
            if constexpr (MODE == kBDisp && SIDE == kCol) {
#pragma unroll
                for (int d = 0; d < DP; ++d)
                    if (d < a.D) o[(int64_t)(w + d) * a.nP] = rKd.get(d);
                w += a.D;
            }
        }
        if constexpr (DO_V) {
#pragma unroll
            for (int c = 0; c < CP; ++c)
                if (c < a.C) o[(int64_t)(w + c) * a.nP] = rKV.get(c);
        }
        return;
    }

    if constexpr (DO_G) {
        if (a.gP) {
            T* g = static_cast<T*>(a.gP) + pi * a.D;
            const bool dist = a.metric != kLinear;
#pragma unroll
            for (int d = 0; d < DP; ++d) {
                if (d < a.D) {
                    T v = rK1.get(d) - (dist ? p[d] * K0.run : T(0));
                    if constexpr (MODE == kBDisp && SIDE == kRow) v -= sumS.run * pv[d];
                    if constexpr (MODE == kBDisp && SIDE == kCol) v += rKd.get(d);
                    g[d] = a.accumulate ? g[d] + v : v;
                }
            }
        }
        if (a.gPb) static_cast<T*>(a.gPb)[pi] = sumH.run;
        if (a.gPw) static_cast<T*>(a.gPw)[pi] = sumHw.run;
    }
    if constexpr (DO_V) {
        if (a.gV) {
            T* gv = static_cast<T*>(a.gV) + pi * a.C;
#pragma unroll
            for (int c = 0; c < CP; ++c)
                if (c < a.C) gv[c] = rKV.get(c);
        }
    }
}

// Sum the per-split partial states of a backward sweep (splits in ascending order) and finalise.
// One thread per (feature, point), points fastest, so every partial-state read is coalesced; the
// feature-0 thread of a point also writes its bias and weight gradients.
template <class T, int MODE, int SIDE, bool DO_G, bool DO_V>
__global__ void __launch_bounds__(kThreads) bwd_merge(const SweepArgs a) {
    griddep_wait();  // launched with launch_pdl: nothing before this touches global memory
    const int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int F = DO_G && DO_V ? (a.D > a.C ? a.D : a.C) : (DO_G ? a.D : a.C);
    if (e >= (int64_t)F * a.nP) return;
    const int f = (int)(e / a.nP);
    const int64_t pi = e - (int64_t)f * a.nP;
    const T* ws = static_cast<const T*>(a.ws);
    const int W = bwd_state_width<MODE, SIDE, DO_G, DO_V>(a.D, a.C);
    const int64_t ss = (int64_t)W * a.nP;
    auto sum = [&](int w) {
        T s = T(0);
        for (int sp = 0; sp < a.splits; ++sp) s += ws[sp * ss + (int64_t)w * a.nP + pi];
        return s;
    };
    int w = 0;
    if constexpr (DO_G) {
        if (f < a.D) {
            if (a.gP) {
                const T* P = static_cast<const T*>(a.P);
                const T* dO = static_cast<const T*>(a.Vp);
                const bool dist = a.metric != kLinear;
                T v = sum(f) - (dist ? P[pi * a.D + f] * sum(a.D) : T(0));
                if (MODE == kBDisp && SIDE == kRow) v -= sum(a.D + 3) * dO[pi * a.D + f];
                if (MODE == kBDisp && SIDE == kCol) v += sum(a.D + 3 + f);
                T* g = static_cast<T*>(a.gP) + pi * a.D + f;
                *g = a.accumulate ? *g + v : v;
            }
            if (f == 0) {
                if (a.gPb) static_cast<T*>(a.gPb)[pi] = sum(a.D + 1);
                if (a.gPw) static_cast<T*>(a.gPw)[pi] = sum(a.D + 2);
            }
        }
        w = a.D + 3 + (MODE == kBDisp ? (SIDE == kRow ? 1 : a.D) : 0);
    }
    if constexpr (DO_V) {
        if (a.gV && f < a.C) static_cast<T*>(a.gV)[pi * a.C + f] = sum(w + f);
    }
}

// ------------------------------------------------------------------------------------------------
// top-k backward: only the selected pairs carry gradient
// ------------------------------------------------------------------------------------------------

// Chain rule of one pair (p own, q other) into the own point's gradient and own parameters.
template <class T>
__device__ __forceinline__ void pair_chain_own(const SweepArgs& a, const T* p, const T* q, T wp, T bp, T wq,
                                               T bq, T G, T* gp, T& gb, T& gw) {
    using E = ExpTraits<T>;
    T dot = T(0), pn = T(0), qn = T(0), d2 = T(0);
    for (int d = 0; d < a.D; ++d) {
        dot = fma(p[d], q[d], dot);
        pn = fma(p[d], p[d], pn);
        qn = fma(q[d], q[d], qn);
        d2 = fma(p[d] - q[d], p[d] - q[d], d2);
    }
    // fp32 distances feature by feature, as in the sweeps (pair_base)
    T base = metric_base<T>(a.metric, dot, pn, qn, T(-a.gamma));
    if (sizeof(T) == 4 && a.metric != kLinear) base = a.metric == kRbf ? ExpTraits<T>::exp(T(-a.gamma) * d2) : d2;
    const T scale = T(a.scale);
    const T t = scale * wp * wq * base + bp + bq;
    const T S = a.apply_exp ? E::exp(t) : t;
    const T H = a.apply_exp ? G * S : G;
    gb += H;
    gw += H * scale * wq * base;
    const T Ev = H * scale * wp * wq;
    const T kappa = a.metric == kLinear ? Ev : (a.metric == kSqeuclidean ? T(-2) * Ev : T(2 * a.gamma) * Ev * base);
    for (int d = 0; d < a.D; ++d) gp[d] += kappa * (q[d] - (a.metric != kLinear ? p[d] : T(0)));
}

// Row side: thread per row i, over its k selected columns.
template <class T>
__global__ void __launch_bounds__(kThreads) topk_bwd_rows(const SweepArgs a, const int64_t* __restrict__ idx,
                                                          const T* __restrict__ gv) {
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= a.nP) return;
    const T* X = static_cast<const T*>(a.P);
    const T* Y = static_cast<const T*>(a.Q);
    T g[64];
    for (int d = 0; d < a.D; ++d) g[d] = T(0);
    T gb = T(0), gw = T(0);
    const T wp = a.pw ? static_cast<const T*>(a.pw)[i] : T(1);
    const T bp = a.pb ? static_cast<const T*>(a.pb)[i] : T(0);
    for (int t = 0; t < a.k; ++t) {
        const int64_t j = idx[i * a.k + t];
        if (j < 0 || j >= a.nQ) continue;
        const T wq = a.qw ? static_cast<const T*>(a.qw)[j] : T(1);
        const T bq = a.qb ? static_cast<const T*>(a.qb)[j] : T(0);
        pair_chain_own<T>(a, X + i * a.D, Y + j * a.D, wp, bp, wq, bq, gv[i * a.k + t], g, gb, gw);
    }
    if (a.gP)
        for (int d = 0; d < a.D; ++d) static_cast<T*>(a.gP)[i * a.D + d] = g[d];
    if (a.gPb) static_cast<T*>(a.gPb)[i] = gb;
    if (a.gPw) static_cast<T*>(a.gPw)[i] = gw;
}

// Column side, step 1: number of selections per column (integer counts: order-independent).
// Indices outside [0, M) are skipped here and in every later step (they carry no gradient).
static __global__ void topk_bwd_count(const int64_t* __restrict__ idx, int64_t n, int64_t M, int* __restrict__ count) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n) return;
    const int64_t j = idx[e];
    if (j >= 0 && j < M) atomicAdd(count + j, 1);
}

// Column side, step 2: exclusive scan of the counts (one CTA of 1024 threads, chunked).
static __global__ void __launch_bounds__(1024) topk_bwd_scan(const int* __restrict__ count, int64_t M, int* __restrict__ start,
                                                      int* __restrict__ cursor) {
    __shared__ int part[1024];
    const int tid = threadIdx.x;
    const int64_t chunk = (M + 1023) / 1024;
    const int64_t lo = tid * chunk, hi = (M < lo + chunk ? M : lo + chunk);
    int s = 0;
    for (int64_t j = lo; j < hi; ++j) s += count[j];
    part[tid] = s;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int v = tid >= off ? part[tid - off] : 0;
        __syncthreads();
        part[tid] += v;
        __syncthreads();
    }
    int run = tid ? part[tid - 1] : 0;
    for (int64_t j = lo; j < hi; ++j) {
        start[j] = run;
        cursor[j] = run;
        run += count[j];
    }
    if (tid == 1023) start[M] = part[1023];
}

// Column side, step 3: place every selection (entry number) into its column's bucket.
static __global__ void topk_bwd_fill(const int64_t* __restrict__ idx, int64_t n, int64_t M, int* __restrict__ cursor,
                              int* __restrict__ bucket) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n) return;
    const int64_t j = idx[e];
    if (j >= 0 && j < M) bucket[atomicAdd(cursor + j, 1)] = (int)e;
}

// Column side, step 4: thread per column; sorts its bucket by entry number (so the sum runs in
// ascending row order whatever order step 3 placed them in) and accumulates the column gradients.
template <class T>
__global__ void __launch_bounds__(kThreads) topk_bwd_cols(const SweepArgs a, const int* __restrict__ start,
                                                          int* __restrict__ bucket, const T* __restrict__ gv) {
    const int64_t j = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (j >= a.nP) return;  // here P = Y (columns), Q = X (rows)
    const int b0 = start[j], b1 = start[j + 1];
    for (int u = b0 + 1; u < b1; ++u) {  // insertion sort of the bucket
        const int v = bucket[u];
        int w = u - 1;
        while (w >= b0 && bucket[w] > v) {
            bucket[w + 1] = bucket[w];
            --w;
        }
        bucket[w + 1] = v;
    }
    const T* Y = static_cast<const T*>(a.P);
    const T* X = static_cast<const T*>(a.Q);
    T g[64];
    for (int d = 0; d < a.D; ++d) g[d] = T(0);
    T gb = T(0), gw = T(0);
    const T wp = a.pw ? static_cast<const T*>(a.pw)[j] : T(1);
    const T bp = a.pb ? static_cast<const T*>(a.pb)[j] : T(0);
    for (int u = b0; u < b1; ++u) {
        const int e = bucket[u];
        const int64_t i = e / a.k;
        const T wq = a.qw ? static_cast<const T*>(a.qw)[i] : T(1);
        const T bq = a.qb ? static_cast<const T*>(a.qb)[i] : T(0);
        pair_chain_own<T>(a, Y + j * a.D, X + i * a.D, wp, bp, wq, bq, gv[e], g, gb, gw);
    }
    if (a.gP)
        for (int d = 0; d < a.D; ++d) {
            T* o = static_cast<T*>(a.gP) + j * a.D + d;
            *o = a.accumulate ? *o + g[d] : g[d];
        }
    if (a.gPb) static_cast<T*>(a.gPb)[j] = gb;
    if (a.gPw) static_cast<T*>(a.gPw)[j] = gw;
}

// ------------------------------------------------------------------------------------------------
// launchers (explicitly instantiated in the inst_*.cu translation units)
// ------------------------------------------------------------------------------------------------

constexpr const char* kFwdNames[] = {"fwd_sweep_matmul", "fwd_sweep_softmax", "fwd_sweep_lse", "fwd_sweep_disp",
                                     "fwd_sweep_svgd"};
constexpr const char* kFwdMergeNames[] = {"fwd_merge_matmul", "fwd_merge_softmax", "fwd_merge_lse", "fwd_merge_disp",
                                          "fwd_merge_svgd"};
// [mode][side][0 = gradients (and dV when fused), 1 = dV only]
constexpr const char* kBwdNames[5][2][2] = {
    {{"bwd_sweep_matmul_row", "bwd_sweep_matmul_row"}, {"bwd_sweep_matmul_col", "bwd_sweep_matmul_col_dv"}},
    {{"bwd_sweep_softmax_row", "bwd_sweep_softmax_row"}, {"bwd_sweep_softmax_col", "bwd_sweep_softmax_col_dv"}},
    {{"bwd_sweep_lse_row", "bwd_sweep_lse_row"}, {"bwd_sweep_lse_col", "bwd_sweep_lse_col"}},
    {{"bwd_sweep_disp_row", "bwd_sweep_disp_row"}, {"bwd_sweep_disp_col", "bwd_sweep_disp_col"}},
    {{"bwd_sweep_lse_sym", "bwd_sweep_lse_sym"}, {"bwd_sweep_lse_sym", "bwd_sweep_lse_sym"}}};
constexpr const char* kBwdMergeNames[5][2] = {{"bwd_merge_matmul_row", "bwd_merge_matmul_col"},
                                              {"bwd_merge_softmax_row", "bwd_merge_softmax_col"},
                                              {"bwd_merge_lse_row", "bwd_merge_lse_col"},
                                              {"bwd_merge_disp_row", "bwd_merge_disp_col"},
                                              {"bwd_merge_lse_sym", "bwd_merge_lse_sym"}};

inline dim3 sweep_grid(const SweepArgs& a) {
    return dim3((unsigned)((a.nP + kThreads - 1) / kThreads), (unsigned)a.splits, 1);
}
inline dim3 row_grid(int64_t n) { return dim3((unsigned)((n + kThreads - 1) / kThreads), 1, 1); }

template <class K>
inline void allow_smem(K* kernel, size_t bytes) {
    if (bytes > 48 * 1024) cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <class T, int DP, int CP, int MODE, bool AFFINE>
void launch_fwd(const SweepArgs& a, cudaStream_t s) {
    constexpr size_t smem = FwdSmem<T, DP, CP, MODE, AFFINE>::bytes;
    allow_smem(fwd_sweep<T, DP, CP, MODE, AFFINE>, smem);
    HookScope h(kFwdNames[MODE], s);
    launch_pdl(fwd_sweep<T, DP, CP, MODE, AFFINE>, sweep_grid(a), dim3(kThreads), smem, s, a);
}
template <class T, int MODE>
void launch_fwd_merge(const SweepArgs& a, cudaStream_t s) {
    HookScope h(kFwdMergeNames[MODE], s);
    launch_pdl(fwd_merge<T, MODE>, row_grid(a.nP), dim3(kThreads), 0, s, a);
}
template <class T, int DP, int K, bool AFFINE>
void launch_topk(const SweepArgs& a, cudaStream_t s) {
    HookScope h("topk_sweep", s);
    launch_pdl(topk_sweep<T, DP, K, AFFINE>, sweep_grid(a), dim3(kThreads), 0, s, a);
}
template <class T, int K>
void launch_topk_merge(const SweepArgs& a, cudaStream_t s) {
    HookScope h("topk_merge", s);
    launch_pdl(topk_merge<T, K>, row_grid(a.nP), dim3(kThreads), 0, s, a);
}
template <class T, int DP, int CP, int MODE, int SIDE, bool DO_G, bool DO_V>
void launch_bwd(const SweepArgs& a, cudaStream_t s) {
    constexpr size_t smem = BwdSmem<T, DP, CP, MODE, SIDE, DO_G, DO_V>::bytes;
    allow_smem(bwd_sweep<T, DP, CP, MODE, SIDE, DO_G, DO_V>, smem);
    HookScope h(kBwdNames[MODE][SIDE][DO_G ? 0 : 1], s);
    launch_pdl(bwd_sweep<T, DP, CP, MODE, SIDE, DO_G, DO_V>, sweep_grid(a), dim3(kThreads), smem, s, a);
}
template <class T, int MODE, int SIDE, bool DO_G, bool DO_V>
void launch_bwd_merge(const SweepArgs& a, cudaStream_t s) {
    const int F = DO_G && DO_V ? (a.D > a.C ? a.D : a.C) : (DO_G ? a.D : a.C);
    HookScope h(kBwdMergeNames[MODE][SIDE], s);
    launch_pdl(bwd_merge<T, MODE, SIDE, DO_G, DO_V>, row_grid((int64_t)F * a.nP), dim3(kThreads), 0, s, a);
}
// rows: P = X, Q = Y; cols: P = Y, Q = X (parameters swapped). count/start/cursor/bucket come from
// the workspace; count must be zero on entry.
template <class T>
void launch_topk_bwd(const SweepArgs& rows, const SweepArgs& cols, const int64_t* idx, const void* gv, int* count,
                     int* start, int* cursor, int* bucket, cudaStream_t s) {
    const T* g = static_cast<const T*>(gv);
    if (rows.gP || rows.gPb || rows.gPw) {
        HookScope h("topk_bwd_rows", s);
        topk_bwd_rows<T><<<row_grid(rows.nP), kThreads, 0, s>>>(rows, idx, g);
    }
    if (cols.gP || cols.gPb || cols.gPw) {
        const int64_t n = rows.nP * (int64_t)rows.k;
        const unsigned nb = (unsigned)((n + 255) / 256);
        {
            HookScope h("topk_bwd_count", s);
            topk_bwd_count<<<nb, 256, 0, s>>>(idx, n, cols.nP, count);
        }
        {
            HookScope h("topk_bwd_scan", s);
            topk_bwd_scan<<<1, 1024, 0, s>>>(count, cols.nP, start, cursor);
        }
        {
            HookScope h("topk_bwd_fill", s);
            topk_bwd_fill<<<nb, 256, 0, s>>>(idx, n, cols.nP, cursor, bucket);
        }
        HookScope h("topk_bwd_cols", s);
        topk_bwd_cols<T><<<row_grid(cols.nP), kThreads, 0, s>>>(cols, start, bucket, g);
    }
}

}  // namespace tp
