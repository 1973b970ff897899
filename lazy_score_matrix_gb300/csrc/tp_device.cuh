// Device-side building blocks shared by every libtp kernel: the canonical score functor held in
// registers, tile staging of the streamed point set into shared memory, and the exp used per pair.
//
// Score (torchpairwise guide "Using Torchpairwise in Models", "Score Expressions"; the rbf kernel
// from "Stein Variational Gradient Descent"):
//   base = |p-q|^2 | p.q | exp(-gamma |p-q|^2);  t = scale*wp*wq*base + bp + bq;  S = exp(t) if asked.
// The metric is symmetric in its two points, so the same functor serves the row sweep (p = x_i,
// q = y_j) and the transposed column sweep (p = y_j, q = x_i), with the row/column parameters
// swapped by the host.
//
// Distances use the norm expansion |p|^2 + |q|^2 - 2 p.q, clamped at 0: one fused multiply-add
// per feature per pair, the same contraction as the linear metric. Norms are computed once per
// owned point and once per staged point.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tp_args.h"

namespace tp {

enum Metric : int { kSqeuclidean = 0, kLinear = 1, kRbf = 2 };

template <class T>
struct Vec16;
template <>
struct Vec16<float> {
    using type = float4;
    static constexpr int n = 4;
};
template <>
struct Vec16<double> {
    using type = double2;
    static constexpr int n = 2;
};

// exp in the working precision. fp32: the hardware base-2 exponential on a pre-scaled argument;
// every fp32 kernel keeps log-sum-exp state in base 2 (kLogB = log2 e) and converts at the end.
// fp64: the CUDA math library's exp (no fp64 special-function unit).
template <class T>
struct ExpTraits;
template <>
struct ExpTraits<float> {
    static constexpr float kLogB = 1.4426950408889634f;  // log2(e)
    static constexpr float kLnB = 0.6931471805599453f;   // ln(2)
    __device__ __forceinline__ static float bexp(float x) {  // 2^x
        float y;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
        return y;
    }
    __device__ __forceinline__ static float blog(float x) { return __log2f(x); }
    __device__ __forceinline__ static float exp(float x) { return bexp(x * kLogB); }
    // The natural log-sum-exp from the base-2 state (max m, sum L of 2^(s - m)): ln2 m + ln L. ln L comes
    // from the accurate logf and ln2 m from a two-term split of ln 2 inside fused multiply-adds, so
    // when the two terms cancel (a log-sum-exp near zero) nothing is lost beyond the final rounding
    // (converting m + log2 L instead loses the ulps of two numbers several times larger than the result).
    __device__ __forceinline__ static float lse(float m, float L) {
        constexpr float kLn2Hi = 0.693147182464599609375f;  // ln 2 rounded to fp32
        constexpr float kLn2Lo = -1.904654323148236e-09f;   // ln 2 - kLn2Hi
        return fmaf(m, kLn2Hi, fmaf(m, kLn2Lo, logf(L)));
    }
};
template <>
struct ExpTraits<double> {
    static constexpr double kLogB = 1.0;
    static constexpr double kLnB = 1.0;
    __device__ __forceinline__ static double bexp(double x) { return ::exp(x); }
    __device__ __forceinline__ static double blog(double x) { return ::log(x); }
    __device__ __forceinline__ static double exp(double x) { return ::exp(x); }
    __device__ __forceinline__ static double lse(double m, double L) { return m + ::log(L); }
};

template <class T>
__device__ __forceinline__ T ninf();
template <>
__device__ __forceinline__ float ninf<float>() {
    return __int_as_float(0xff800000);
}
template <>
__device__ __forceinline__ double ninf<double>() {
    return __longlong_as_double(0xfff0000000000000ULL);
}
template <class T>
__device__ __forceinline__ T pinf();
template <>
__device__ __forceinline__ float pinf<float>() {
    return __int_as_float(0x7f800000);
}
template <>
__device__ __forceinline__ double pinf<double>() {
    return __longlong_as_double(0x7ff0000000000000ULL);
}

// Dot product of a register-resident point with a shared-memory row (16-byte aligned, padded
// with zeros to DP). Uses 16-byte broadcast loads and Vec16<T>::n independent FMA chains.
template <class T, int DP>
__device__ __forceinline__ T dot_regs_smem(const T (&p)[DP], const T* __restrict__ q) {
    using V = typename Vec16<T>::type;
    constexpr int VN = Vec16<T>::n;
    static_assert(DP % VN == 0, "padded width must be a multiple of the vector width");
    T acc[VN];
#pragma unroll
    for (int u = 0; u < VN; ++u) acc[u] = T(0);
#pragma unroll
    for (int d = 0; d < DP; d += VN) {
        V v = *reinterpret_cast<const V*>(q + d);
        if constexpr (VN == 4) {
            acc[0] = fma(p[d + 0], v.x, acc[0]);
            acc[1] = fma(p[d + 1], v.y, acc[1]);
            acc[2] = fma(p[d + 2], v.z, acc[2]);
            acc[3] = fma(p[d + 3], v.w, acc[3]);
        } else {
            acc[0] = fma(p[d + 0], v.x, acc[0]);
            acc[1] = fma(p[d + 1], v.y, acc[1]);
        }
    }
    if constexpr (VN == 4) return (acc[0] + acc[1]) + (acc[2] + acc[3]);
    else return acc[0] + acc[1];
}

// acc[c] += w * q[c] over a shared-memory row (broadcast 16-byte loads).
template <class T, int CP>
__device__ __forceinline__ void axpy_smem(T (&acc)[CP], T w, const T* __restrict__ q) {
    using V = typename Vec16<T>::type;
    constexpr int VN = Vec16<T>::n;
#pragma unroll
    for (int c = 0; c < CP; c += VN) {
        V v = *reinterpret_cast<const V*>(q + c);
        if constexpr (VN == 4) {
            acc[c + 0] = fma(w, v.x, acc[c + 0]);
            acc[c + 1] = fma(w, v.y, acc[c + 1]);
            acc[c + 2] = fma(w, v.z, acc[c + 2]);
            acc[c + 3] = fma(w, v.w, acc[c + 3]);
        } else {
            acc[c + 0] = fma(w, v.x, acc[c + 0]);
            acc[c + 1] = fma(w, v.y, acc[c + 1]);
        }
    }
}

// Copy rows [row0, row0+cnt) of a row-major [*, W] global array into a [kTile][WP] shared tile.
// Positions W..WP-1 of each row are never written (the caller zeroes them once). `vec` selects
// 16-byte loads, valid when W == WP and the source is 16-byte aligned.
template <class T, int WP>
__device__ __forceinline__ void stage_rows(T* __restrict__ s, const T* __restrict__ g, int64_t row0,
                                           int cnt, int W, bool vec) {
    if (vec) {
        using V = typename Vec16<T>::type;
        constexpr int VN = Vec16<T>::n;
        const V* src = reinterpret_cast<const V*>(g + row0 * WP);
        V* dst = reinterpret_cast<V*>(s);
        const int total = cnt * (WP / VN);
        for (int e = threadIdx.x; e < total; e += kThreads) dst[e] = __ldg(src + e);
    } else {
        const T* src = g + row0 * W;
        const int total = cnt * W;
        for (int e = threadIdx.x; e < total; e += kThreads) {
            const int r = e / W;
            const int d = e - r * W;
            s[r * WP + d] = __ldg(src + e);
        }
    }
}

// Copy a per-point scalar array slice into shared memory; `fill` where the array is absent.
template <class T>
__device__ __forceinline__ void stage_scalar(T* __restrict__ s, const T* __restrict__ g, int64_t row0,
                                             int cnt, T fill) {
    for (int e = threadIdx.x; e < cnt; e += kThreads) s[e] = g ? __ldg(g + row0 + e) : fill;
}

template <class T>
__device__ __forceinline__ void zero_smem(T* s, int n) {
    for (int e = threadIdx.x; e < n; e += kThreads) s[e] = T(0);
}

// Load a point into registers (zero-padded to DP); `valid` false gives zeros.
template <class T, int DP>
__device__ __forceinline__ void load_point(T (&p)[DP], const T* __restrict__ g, int64_t idx, int D,
                                           bool valid) {
#pragma unroll
    for (int d = 0; d < DP; ++d) p[d] = (valid && d < D) ? __ldg(g + idx * D + d) : T(0);
}

template <class T, int DP>
__device__ __forceinline__ T sqnorm(const T (&p)[DP]) {
    T a = T(0);
#pragma unroll
    for (int d = 0; d < DP; ++d) a = fma(p[d], p[d], a);
    return a;
}

// Squared norms of the staged rows (one thread per row).
template <class T, int DP>
__device__ __forceinline__ void stage_norms(T* __restrict__ sn, const T* __restrict__ sq, int cnt) {
    for (int r = threadIdx.x; r < cnt; r += kThreads) {
        T a = T(0);
#pragma unroll
        for (int d = 0; d < DP; ++d) a = fma(sq[r * DP + d], sq[r * DP + d], a);
        sn[r] = a;
    }
}

// The metric value from the dot product and both squared norms.
template <class T>
__device__ __forceinline__ T metric_base(int metric, T dot, T pn, T qn, T neg_gamma) {
    if (metric == kLinear) return dot;
    T d2 = fmax(fma(T(-2), dot, pn + qn), T(0));
    if (metric == kRbf) return ExpTraits<T>::exp(neg_gamma * d2);
    return d2;
}

// |p - q|^2 of a register-resident point and a shared-memory row (both zero-padded to DP), feature by
// feature: 16-byte broadcast loads, Vec16<T>::n independent FMA chains.
template <class T, int DP>
__device__ __forceinline__ T dist2_regs_smem(const T (&p)[DP], const T* __restrict__ q) {
    using V = typename Vec16<T>::type;
    constexpr int VN = Vec16<T>::n;
    T acc[VN];
#pragma unroll
    for (int u = 0; u < VN; ++u) acc[u] = T(0);
#pragma unroll
    for (int d = 0; d < DP; d += VN) {
        V v = *reinterpret_cast<const V*>(q + d);
        if constexpr (VN == 4) {
            const T e0 = p[d + 0] - v.x, e1 = p[d + 1] - v.y, e2 = p[d + 2] - v.z, e3 = p[d + 3] - v.w;
            acc[0] = fma(e0, e0, acc[0]);
            acc[1] = fma(e1, e1, acc[1]);
            acc[2] = fma(e2, e2, acc[2]);
            acc[3] = fma(e3, e3, acc[3]);
        } else {
            const T e0 = p[d + 0] - v.x, e1 = p[d + 1] - v.y;
            acc[0] = fma(e0, e0, acc[0]);
            acc[1] = fma(e1, e1, acc[1]);
        }
    }
    if constexpr (VN == 4) return (acc[0] + acc[1]) + (acc[2] + acc[3]);
    else return acc[0] + acc[1];
}

// The metric value of a register-resident point p and a staged row q (pn, qn: their squared norms).
// Linear: the dot product. Distance metrics in fp32 subtract feature by feature: the expansion
// |p|^2 + |q|^2 - 2 p.q rounds at the size of |p|^2 + |q|^2, so a distance much smaller than the
// points' norms keeps only the bits the cancellation leaves (several fp32 ulps of |p|^2 + |q|^2, which
// a log-sum-exp or softmax of the scores then carries). fp64 keeps the expansion (one FMA per feature
// instead of two): its cancellation error stays far below the fp64 tolerance. Exact either way on
// integer-valued points whose squared norms are below 2^24 (top-k's exact tie order).
template <class T, int DP>
__device__ __forceinline__ T pair_base(int metric, const T (&p)[DP], const T* __restrict__ q, T pn, T qn,
                                       T neg_gamma) {
    if (metric == kLinear) return dot_regs_smem<T, DP>(p, q);
    T d2;
    if constexpr (sizeof(T) == 4) d2 = dist2_regs_smem<T, DP>(p, q);
    else d2 = fmax(fma(T(-2), dot_regs_smem<T, DP>(p, q), pn + qn), T(0));
    if (metric == kRbf) return ExpTraits<T>::exp(neg_gamma * d2);
    return d2;
}

// Insert (key, idx) into the sorted list when it beats the last entry. Entries of equal key keep
// their order, so streaming indices in ascending order gives ascending indices among ties.
template <class T, int K>
__device__ __forceinline__ void topk_insert(T (&kv)[K], int (&ki)[K], T key, int idx) {
    if (!(key < kv[K - 1])) return;
    bool placed = false;
#pragma unroll
    for (int t = K - 1; t > 0; --t) {
        const bool shift = kv[t - 1] > key;
        if (!placed) {
            kv[t] = shift ? kv[t - 1] : key;
            ki[t] = shift ? ki[t - 1] : idx;
            placed = !shift;
        }
    }
    if (!placed) {
        kv[0] = key;
        ki[0] = idx;
    }
}

// Lexicographic (key, index) insertion, used where candidates arrive out of index order.
template <class T, int K>
__device__ __forceinline__ void topk_insert_lex(T (&kv)[K], int (&ki)[K], T key, int idx) {
    auto less = [](T av, int ai, T bv, int bi) { return av < bv || (av == bv && ai < bi); };
    if (!less(key, idx, kv[K - 1], ki[K - 1])) return;
    bool placed = false;
#pragma unroll
    for (int t = K - 1; t > 0; --t) {
        const bool shift = less(key, idx, kv[t - 1], ki[t - 1]);
        if (!placed) {
            kv[t] = shift ? kv[t - 1] : key;
            ki[t] = shift ? ki[t - 1] : idx;
            placed = !shift;
        }
    }
    if (!placed) {
        kv[0] = key;
        ki[0] = idx;
    }
}

}  // namespace tp
