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

// Programmatic dependent launch (kernels started with launch_pdl, tp_launch.h): such a kernel may begin
// while the kernel before it on the stream is still running. griddep_wait returns once that grid has
// completed and its memory operations are visible, so nothing before it may read or write global memory;
// griddep_launch lets the next such kernel on the stream begin its prologue. In a kernel launched without
// the attribute both are no-ops.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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
// fp64: exp_table below (no fp64 special-function unit).
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
// 2^(j/64), j = 0..63, each correctly rounded to fp64 (computed in 60-digit decimal arithmetic; a CPU test
// recomputes every entry).
static __device__ const double kExp2Tab64[64] = {
    0x1.0000000000000p+0, 0x1.02c9a3e778061p+0, 0x1.059b0d3158574p+0, 0x1.0874518759bc8p+0,
    0x1.0b5586cf9890fp+0, 0x1.0e3ec32d3d1a2p+0, 0x1.11301d0125b51p+0, 0x1.1429aaea92de0p+0,
    0x1.172b83c7d517bp+0, 0x1.1a35beb6fcb75p+0, 0x1.1d4873168b9aap+0, 0x1.2063b88628cd6p+0,
    0x1.2387a6e756238p+0, 0x1.26b4565e27cddp+0, 0x1.29e9df51fdee1p+0, 0x1.2d285a6e4030bp+0,
    0x1.306fe0a31b715p+0, 0x1.33c08b26416ffp+0, 0x1.371a7373aa9cbp+0, 0x1.3a7db34e59ff7p+0,
    0x1.3dea64c123422p+0, 0x1.4160a21f72e2ap+0, 0x1.44e086061892dp+0, 0x1.486a2b5c13cd0p+0,
    0x1.4bfdad5362a27p+0, 0x1.4f9b2769d2ca7p+0, 0x1.5342b569d4f82p+0, 0x1.56f4736b527dap+0,
    0x1.5ab07dd485429p+0, 0x1.5e76f15ad2148p+0, 0x1.6247eb03a5585p+0, 0x1.6623882552225p+0,
    0x1.6a09e667f3bcdp+0, 0x1.6dfb23c651a2fp+0, 0x1.71f75e8ec5f74p+0, 0x1.75feb564267c9p+0,
    0x1.7a11473eb0187p+0, 0x1.7e2f336cf4e62p+0, 0x1.82589994cce13p+0, 0x1.868d99b4492edp+0,
    0x1.8ace5422aa0dbp+0, 0x1.8f1ae99157736p+0, 0x1.93737b0cdc5e5p+0, 0x1.97d829fde4e50p+0,
    0x1.9c49182a3f090p+0, 0x1.a0c667b5de565p+0, 0x1.a5503b23e255dp+0, 0x1.a9e6b5579fdbfp+0,
    0x1.ae89f995ad3adp+0, 0x1.b33a2b84f15fbp+0, 0x1.b7f76f2fb5e47p+0, 0x1.bcc1e904bc1d2p+0,
    0x1.c199bdd85529cp+0, 0x1.c67f12e57d14bp+0, 0x1.cb720dcef9069p+0, 0x1.d072d4a07897cp+0,
    0x1.d5818dcfba487p+0, 0x1.da9e603db3285p+0, 0x1.dfc97337b9b5fp+0, 0x1.e502ee78b3ff6p+0,
    0x1.ea4afa2a490dap+0, 0x1.efa1bee615a27p+0, 0x1.f50765b6e4540p+0, 0x1.fa7c1819e90d8p+0,
};

// fp64 exp by the table-driven method of P. T. P. Tang ("Table-driven implementation of the exponential
// function in IEEE floating-point arithmetic", ACM Trans. Math. Softw. 15(2), 1989): with N the integer
// nearest x 64/ln2, x = N ln2/64 + r, |r| <= ln2/128, and exp(x) = 2^(N >> 6) 2^((N & 63)/64) e^r.
// 2^(j/64) comes from the table above, e^r - 1 from its degree-5 Taylor polynomial (the first omitted
// term r^6/720 is below 4e-17 relative for |r| <= ln2/128), and r from a two-part ln2/64 whose leading
// part has 36 significant bits, so N L1 is exact for every N that occurs. About ten fp64 operations
// (a general library exp takes about twice as many, on a pipe the fp64 sweeps saturate). Arguments
// below -707 give 0 (exp(-707) ~ 1e-307: a term that small changes no fp64 sum of larger ones); above
// 709.78, +inf; NaN is not handled (non-finite inputs are unsupported).
__device__ __forceinline__ double exp_table(double x) {
    constexpr double kInvL = 0x1.71547652b82fep+6;                            // 64 / ln 2
    constexpr double kL1 = 0x1.62e42fefa0000p-7, kL2 = 0x1.cf79abc9e3b3ap-46;  // ln2/64 = L1 + L2
    constexpr double kShift = 0x1.8p52;  // adding 1.5 2^52 rounds to an integer kept in the low word
    // one compare per bound, shared by the clamp and the result (fmin/fmax would compare again)
    const bool under = x < -707.0, over = x > 709.78;
    const double xc = under ? -707.0 : (over ? 709.78 : x);
    const double s = fma(xc, kInvL, kShift);
    const int N = __double2loint(s);
    const double Nd = s - kShift;
    const double r = fma(-Nd, kL2, fma(-Nd, kL1, xc));
    const double q = fma(r, fma(r, fma(r, 1.0 / 120.0, 1.0 / 24.0), 1.0 / 6.0), 0.5);
    const double t = __ldg(kExp2Tab64 + (N & 63));
    const double y = fma(t, fma(r * r, q, r), t);  // 2^(j/64) e^r, in [0.99, 1.99]
    // times 2^(N >> 6), N >> 6 in [-1020, 1023]: added to the exponent field (the result stays normal)
    const double res = __hiloint2double(__double2hiint(y) + (int)((unsigned)(N >> 6) << 20), __double2loint(y));
    return under ? 0.0 : (over ? __longlong_as_double(0x7ff0000000000000ULL) : res);
}

template <>
struct ExpTraits<double> {
    static constexpr double kLogB = 1.0;
    static constexpr double kLnB = 1.0;
    __device__ __forceinline__ static double bexp(double x) { return exp_table(x); }
    __device__ __forceinline__ static double blog(double x) { return ::log(x); }
    __device__ __forceinline__ static double exp(double x) { return exp_table(x); }
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
    else d2 = fma(T(-2), dot_regs_smem<T, DP>(p, q), pn + qn);  // the norm expansion may round below 0
    // rbf needs no clamp (a d2 a rounding below 0 gives exp 1 + O(eps)); in fp64 the compare it saves
    // runs on the FP64 pipe that bounds the sweep
    if (metric == kRbf) return ExpTraits<T>::exp(neg_gamma * d2);
    return sizeof(T) == 4 ? d2 : fmax(d2, T(0));
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
