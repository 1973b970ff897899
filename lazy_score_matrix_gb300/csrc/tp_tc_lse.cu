// Row log-sum-exp and its symmetric backward on the Blackwell tensor cores (fp32 data, D = 64
// features, no row/column parameters): torchpairwise guide "Using Torchpairwise in Models", Task Map
// (InfoNCE row: S.logsumexp(-1, exclude_self=True) on S = lazy(z, z, "linear") / t) and Score
// Expressions; the backward re-evaluates the tiles (introduction, on first derivatives).
//
// Operands. Each point row x is scaled by a power of two 2^e (e per row, chosen so max|x| * 2^e lies in
// [2^14, 2^15)) and split into two fp16 values, hi = fp16(x 2^e) and lo = fp16(x 2^e - hi), both rounded
// to nearest: 11 + 11 significant bits, like a tf32 hi/lo split, at half the bytes and with K = 16 per
// tcgen05.mma kind::f16 instead of 8. The power of two keeps every element that matters in fp16's
// normal range whatever the data's scale, and is undone exactly on the fp32 result. A dot product is
// x.y ~ (xh.yh + (xh.yl + xl.yh)) 2^-(e_x + e_y): hi*hi accumulates in TMEM columns of its own and the
// two small products together, and the epilogue adds the two in fp32 (the accumulator truncates
// toward zero after each MMA; keeping hi*hi apart keeps the small products' bits).
//
// Schedule. Persistent CTAs, one per SM: the (row block, column tile) pairs are numbered row-block major
// and cut into equal contiguous ranges, one per CTA. Warp 0 lane 0 loads tiles with TMA (128-byte
// swizzle), warp 1 owns the TMEM allocation and its lane 0 issues the MMAs, the other warps are the
// epilogue (one row per thread, four warps per TMEM lane quarter). A CTA writes a partial per row for
// each row block it touched; the last CTA to finish a row block (an atomic count per row block) adds
// the partials of its rows in CTA order, so results are deterministic.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tp_args.h"
#include "tp_device.cuh"
#include "tp_launch.h"
#include "tp_tc.cuh"
#include "tp_tc_host.h"

namespace tp {
namespace tc {

constexpr int kBM = 128;                    // rows per tile (TMEM lanes)
constexpr int kRowBytes = 128;              // one point: 64 fp16 features
constexpr int kHalfTile = kBM * kRowBytes;  // 128 rows of hi (or lo): 16 KB
constexpr int kEpi = 16;                    // epilogue warps: 4 per TMEM lane quarter
constexpr int kTcThreads = 32 * (2 + kEpi);
constexpr int kGrid = 152;                  // persistent CTAs: one per GB300 SM

// Base-2 score of one element from its dot product (metric, scale, exp).
template <int METRIC, bool EXP>
__device__ __forceinline__ float score2(float dot, float xn, float yn, float scale, float neg_gamma_log2) {
    constexpr float kL2E = 1.4426950408889634f;
    float base;
    if (METRIC == kLinear) {
        base = dot;
    } else {
        const float d2 = fmaxf(fmaf(-2.f, dot, xn + yn), 0.f);
        base = METRIC == kRbf ? ExpTraits<float>::bexp(neg_gamma_log2 * d2) : d2;
    }
    const float t = scale * base;
    const float S = EXP ? ExpTraits<float>::bexp(t * kL2E) : t;
    return S * kL2E;
}

// Per point row: the fp16 hi/lo split of x 2^e, 2^-e, and |x|^2. One warp per row, two features per
// lane. rows: rows of x; rows_pad: rows of inv_scale and norm (zeros past rows); cnt (optional): ncnt
// counters zeroed for the kernel that follows (ncnt <= rows_pad).
__global__ void __launch_bounds__(256) tc_split16(const float* __restrict__ x, int64_t rows, int64_t rows_pad,
                                                  __half2* __restrict__ hi, __half2* __restrict__ lo,
                                                  float* __restrict__ inv_scale, float* __restrict__ norm,
                                                  int* __restrict__ cnt, int64_t ncnt) {
    griddep_wait();
    griddep_launch();
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (cnt && lane == 0 && r < ncnt) cnt[r] = 0;  // the main kernel's per-row-block arrival counters
    if (r >= rows_pad) return;
    if (r >= rows) {
        if (lane == 0) {
            inv_scale[r] = 0.f;
            norm[r] = 0.f;
        }
        return;
    }
    const float2 v = reinterpret_cast<const float2*>(x + r * 64)[lane];
    float m = fmaxf(fabsf(v.x), fabsf(v.y)), ss = fmaf(v.x, v.x, v.y * v.y);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    }
    const int e = f16_row_exponent(m);
    const float f = pow2i(e);
    const float a = v.x * f, b = v.y * f;
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    hi[r * 32 + lane] = h;
    lo[r * 32 + lane] = __floats2half2_rn(a - hf.x, b - hf.y);
    if (lane == 0) {
        inv_scale[r] = pow2i(-e);
        norm[r] = ss;
    }
}

void launch_split16(const float* x, int64_t rows, int64_t rows_pad, void* hi, void* lo, float* inv_scale, float* norm,
                    int* cnt, int64_t ncnt, cudaStream_t s) {
    HookScope h("tc_split16", s);
    launch_pdl(tc_split16, dim3((unsigned)((rows_pad + 7) / 8)), dim3(256), 0, s, x, rows, rows_pad,
               static_cast<__half2*>(hi), static_cast<__half2*>(lo), inv_scale, norm, cnt, ncnt);
}

// ------------------------------------------------------------------------------------------------
// Forward: 128 x 128 tiles. Per K step of 16 features: Xh [Yh; Yl] (N = 256: hi*hi into accumulator
// columns 0..127, hi*lo into 128..255), then Xl Yh (N = 128) into 128..255. Two accumulators of 256
// columns, so the MMAs of tile i+1 overlap the epilogue of tile i; four B stages of 32 KB.
// ------------------------------------------------------------------------------------------------
constexpr int kBN = 128;                 // columns per forward tile
constexpr int kStagesF = 4;
constexpr int kPairF = 2 * kHalfTile;    // hi + lo of 128 points: 32 KB
constexpr size_t kSmemF = (size_t)kPairF * (1 + kStagesF) + 256 + 1024;
static_assert(kSmemF <= 232448, "dynamic shared memory per CTA");

struct LseTcParams {
    int64_t N, M;
    Sched sc;    // the tiles each row block streams (all CT of them without a pair mask)
    int64_t T;   // total tiles
    int G;       // CTAs
    int metric, apply_exp, exclude_self, same;
    float scale;
    float neg_gamma_log2;  // -gamma * log2(e)
    const float* xs;       // 2^-e of each row point
    const float* ys;       // 2^-e of each column point
    const float* xn;       // |x_i|^2 (distance metrics)
    const float* yn;       // |y_j|^2
    float* part;           // [RB + G][4 column parts][2][128] partial (max, sum) in base 2: slot position + CTA
    int* cnt;              // [RB] CTAs done with each row block (zeroed by the split pre-pass)
    float* lse;            // [N] output
    int* err;
    // after lse_fwd_sym_tc (null otherwise): sym[0] == 0 means that sweep covered the rows and this kernel
    // only merges its partials (prow, pcol; Gs its CTAs) before anything else; 1 means it sweeps as usual
    const int* sym;
    const float* prow;
    const float* pcol;
    int Gs;
};

// lse of row `row` of row block rb from the partials of every CTA that saw it, in CTA order (one
// pass, combining the (max, sum) pairs online in a fixed order: the result does not depend on timing).
__device__ __noinline__ float lse_merge_row(const LseTcParams& p, int rb, int lr) {
    const int64_t v = sched_pos(p.sc, rb), t0 = tile_start(p.sc, v), t1 = tile_start(p.sc, v + 1) - 1;
    const int c_lo = cta_of_tile(p.T, p.G, t0), c_hi = cta_of_tile(p.T, p.G, t1);
    float m = ninf<float>(), l = 0.f;
    for (int c = c_lo; c <= c_hi; ++c) {
        const float* o = p.part + ((size_t)((v + c) * 4) * 2) * kBM + lr;
        float pm[4], pl[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            pm[h] = __ldcg(o + (size_t)h * 2 * kBM);
            pl[h] = __ldcg(o + (size_t)h * 2 * kBM + kBM);
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            if (pm[h] == ninf<float>()) continue;
            if (pm[h] > m) {
                l = l * ExpTraits<float>::bexp(m - pm[h]) + pl[h];
                m = pm[h];
            } else {
                l += pl[h] * ExpTraits<float>::bexp(pm[h] - m);
            }
        }
    }
    return l > 0.f ? ExpTraits<float>::lse(m, l) : ninf<float>();
}

// lse of rows from the triangle sweep's partials (lse_fwd_tc in merge mode): eight threads per row, each
// adding every eighth term (the row partials of the CTAs that swept the row's block, in CTA order, then the
// column partials of the tiles (I, R), I < R, in order of I), the eight sums combined in a fixed tree.
__device__ __noinline__ void sym_merge(const LseTcParams& p) {
    const int RB = (int)((p.N + kBM - 1) / kBM);
    const int64_t T = (int64_t)RB * (RB + 1) / 2;
    const float M = __int_as_float(__ldcg(p.sym + 1));
    const int64_t wpb = blockDim.x >> 5, lane = threadIdx.x & 31;
    for (int64_t base = ((int64_t)blockIdx.x * wpb + (threadIdx.x >> 5)) * 4; base < p.N;
         base += (int64_t)gridDim.x * wpb * 4) {  // warp-uniform: four rows per warp, eight lanes per row
        const int64_t row = base + (lane >> 3);
        const int k = (int)(lane & 7);
        float l = 0.f;
        if (row < p.N) {
            const int R = (int)(row / kBM), lr = (int)(row % kBM);
            const int64_t t0 = sym_start(R, RB);
            const int c_lo = cta_of_tile(T, p.Gs, t0), c_hi = cta_of_tile(T, p.Gs, t0 + (RB - R) - 1);
            const int nrow = c_hi - c_lo + 1, nterm = nrow + R;
            for (int m0 = k; m0 < nterm; m0 += 32) {  // four independent loads in flight, added in order
                float4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int m = m0 + 8 * u;
                    const float* src = m < nrow ? p.prow + ((size_t)(R + c_lo + m) * kBM + lr) * 4
                                                : p.pcol + ((size_t)(sym_start(m - nrow, RB) + R - (m - nrow)) * kBM + lr) * 4;
                    v[u] = m < nterm ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) l += (v[u].x + v[u].y) + (v[u].z + v[u].w);
            }
        }
        l += __shfl_down_sync(0xffffffffu, l, 1, 8);
        l += __shfl_down_sync(0xffffffffu, l, 2, 8);
        l += __shfl_down_sync(0xffffffffu, l, 4, 8);
        if (k == 0 && row < p.N) p.lse[row] = l > 0.f ? ExpTraits<float>::lse(M, l) : ninf<float>();
    }
}

template <int METRIC, bool EXP>
__global__ void __launch_bounds__(kTcThreads, 1)
    lse_fwd_tc(const __grid_constant__ CUtensorMap mXh, const __grid_constant__ CUtensorMap mXl,
               const __grid_constant__ CUtensorMap mYh, const __grid_constant__ CUtensorMap mYl, const LseTcParams p) {
    if (p.sym) {  // after the triangle sweep: merge its partials, unless it fell back
        griddep_wait();
        if (__ldcg(p.sym) == 0) {
            griddep_launch();
            sym_merge(p);
            return;
        }
    }
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_base1024(smem_raw);
    unsigned char* sA = sm;               // [hi 128 rows | lo 128 rows]
    unsigned char* sB = sm + kPairF;      // stage s at sB + s * kPairF: [hi 128 points | lo 128 points]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + (size_t)kPairF * (1 + kStagesF));
    uint64_t* a_full = bars + 0;
    uint64_t* a_empty = bars + 1;
    uint64_t* b_full = bars + 2;                 // [kStagesF]
    uint64_t* b_empty = b_full + kStagesF;       // [kStagesF]
    uint64_t* acc_full = b_empty + kStagesF;     // [2]
    uint64_t* acc_empty = acc_full + 2;          // [2]
    uint64_t* fl_bar = acc_empty + 2;            // the epilogue wrote its partials of a row block
    uint64_t* dec_bar = fl_bar + 1;              // the CTA knows whether it merges that row block
    uint32_t* tslot = reinterpret_cast<uint32_t*>(dec_bar + 1);
    volatile int* sflag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t_begin = range_start(p.T, p.G, blockIdx.x), t_end = range_start(p.T, p.G, blockIdx.x + 1);

    if (threadIdx.x == 0) {
        prefetch_map(&mXh);
        prefetch_map(&mXl);
        prefetch_map(&mYh);
        prefetch_map(&mYl);
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int s = 0; s < kStagesF; ++s) {
            mbar_init(b_full + s, 1);
            mbar_init(b_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, kEpi);  // one arrival per epilogue warp
        }
        mbar_init(fl_bar, kEpi);
        mbar_init(dec_bar, 1);
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    griddep_wait();
    griddep_launch();

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            SchedCursor cur(p.sc, t_begin);
            for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next(p.sc)) {
                const int64_t i = t - t_begin;
                const int rb = cur.rb, ct = cur.ct;
                if (rb != rb_cur) {
                    if (a_uses > 0) ok = mbar_wait(a_empty, (a_uses - 1) & 1, p.err, 11);
                    if (!ok) break;
                    mbar_expect_tx(a_full, kPairF);
                    tma_load_2d(sA, &mXh, 0, rb * kBM, a_full);
                    tma_load_2d(sA + kHalfTile, &mXl, 0, rb * kBM, a_full);
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStagesF), r = (int)(i / kStagesF);
                if (r >= 1) ok = mbar_wait(b_empty + s, (r - 1) & 1, p.err, 12);
                if (!ok) break;
                unsigned char* dst = sB + (size_t)s * kPairF;
                mbar_expect_tx(b_full + s, kPairF);
                tma_load_2d(dst, &mYh, 0, ct * kBN, b_full + s);
                tma_load_2d(dst + kHalfTile, &mYl, 0, ct * kBN, b_full + s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            constexpr uint32_t id256 = idesc_f16(kBM, 2 * kBN, false);
            constexpr uint32_t id128 = idesc_f16(kBM, kBN, false);
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            SchedCursor cur(p.sc, t_begin);
            for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next(p.sc)) {
                const int64_t i = t - t_begin;
                const int rb = cur.rb;
                if (rb != rb_cur) {
                    if (a_uses > 0) mma_commit(a_empty);  // the previous A is free once its MMAs finish
                    ok = mbar_wait(a_full, a_uses & 1, p.err, 13);
                    if (!ok) break;
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStagesF), r = (int)(i / kStagesF), b = (int)(i & 1), rr = (int)(i >> 1);
                ok = mbar_wait(b_full + s, r & 1, p.err, 14);
                if (ok && rr >= 1) ok = mbar_wait(acc_empty + b, (rr - 1) & 1, p.err, 15);
                if (!ok) break;
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * 256);
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB + (size_t)s * kPairF);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ko = (uint32_t)(ks * 32);
                    mma_f16(d, desc_sw128(a0 + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), id256, ks > 0 ? 1u : 0u);
                    mma_f16(d + 128, desc_sw128(a0 + kHalfTile + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), id128,
                            1u);
                }
                mma_commit(b_empty + s);
                mma_commit(acc_full + b);
            }
        }
    } else {  // ---------------- epilogue: one row per thread, 32 of the tile's columns per warp
        constexpr float kL2E = 1.4426950408889634f;
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int sub = (warp - 2) >> 2;        // columns [32 sub, 32 sub + 32) of each tile
        const int lr = q * 32 + lane;           // row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(sub * 32);
        int rb_cur = -1, seg = 0;
        float m = ninf<float>(), l = 0.f, xn = 0.f, c1r = 0.f, xs = 0.f;
        bool ok = true;
        const int etid = threadIdx.x - 64;  // 0 .. 32 kEpi - 1
        // Write this thread's partial of row block rb_cur. The CTA that completes the row block (the last
        // of the CTAs whose tile ranges meet it to count itself in) merges its rows into lse.
        auto flush = [&]() {
            const int64_t v = sched_pos(p.sc, rb_cur);
            float* o = p.part + ((size_t)((v + blockIdx.x) * 4 + sub) * 2) * kBM;
            o[lr] = m;
            o[kBM + lr] = l;
            __threadfence();
            mbar_arrive_warp(fl_bar);
            if (etid == 0) {
                int last = 0;
                if (mbar_wait(fl_bar, (uint32_t)(seg & 1), p.err, 17)) {
                    const int64_t t0 = tile_start(p.sc, v), t1 = tile_start(p.sc, v + 1) - 1;
                    const int need = cta_of_tile(p.T, p.G, t1) - cta_of_tile(p.T, p.G, t0) + 1;
                    last = atomicAdd(p.cnt + rb_cur, 1) + 1 == need;
                    __threadfence();
                }
                *sflag = last;
                mbar_arrive(dec_bar);
            }
            if (mbar_wait(dec_bar, (uint32_t)(seg & 1), p.err, 18) && *sflag && etid < kBM) {
                const int64_t r = (int64_t)rb_cur * kBM + etid;
                if (r < p.N) p.lse[r] = lse_merge_row(p, rb_cur, etid);
            }
            ++seg;
        };
        SchedCursor cur(p.sc, t_begin);
        for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next(p.sc)) {
            const int64_t i = t - t_begin;
            const int rb = cur.rb, ct = cur.ct;
            const int64_t row = (int64_t)rb * kBM + lr;
            if (rb != rb_cur) {
                if (rb_cur >= 0) flush();
                m = ninf<float>();
                l = 0.f;
                rb_cur = rb;
                const bool live = row < p.N;
                xn = (METRIC != kLinear && live) ? p.xn[row] : 0.f;
                xs = live ? p.xs[row] : 0.f;
                c1r = p.scale * kL2E * xs;
            }
            const int b = (int)(i & 1), rr = (int)(i >> 1);
            ok = mbar_wait_warp(acc_full + b, rr & 1, p.err, 16);
            if (!ok) break;
            fence_after_sync();
            float v[32];  // hi*hi + (hi*lo + lo*hi), 16 columns at a time to bound live registers
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                float t0[16], t1[16];
                tmem_ld16x2(lane_base + (uint32_t)(b * 256 + hlf * 16), lane_base + (uint32_t)(b * 256 + 128 + hlf * 16),
                            t0, t1);
#pragma unroll
                for (int u = 0; u < 16; ++u) v[hlf * 16 + u] = t0[u] + t1[u];
            }
            fence_before_sync();
            mbar_arrive_warp(acc_empty + b);  // the values are in registers: the MMA may reuse the buffer
            const int64_t j0 = (int64_t)ct * kBN + sub * 32;
            const bool diag = row >= j0 && row < j0 + 32;
            // a pair mask cuts into these 32 columns (the first or the last of them is outside it)
            const bool cut = p.sc.pm != 0 &&
                             !(pair_in(p.sc.pm, p.sc.band, row, j0) && pair_in(p.sc.pm, p.sc.band, row, j0 + 31));
            const bool masked = p.M - j0 < 32 || cut || (diag && (p.exclude_self || (p.same && METRIC != kLinear)));
            const float4* ys4 = reinterpret_cast<const float4*>(p.ys + j0);  // padded: 32 readable entries
            if (METRIC == kLinear && !EXP && !masked && c1r > 0.f) {
                // common case: score c1r * (x.y 2^(e_x+e_y)) 2^-e_y with c1r = scale log2(e) 2^-e_x > 0. The
                // row factor commutes with the max and folds into the exp's FMA.
#pragma unroll
                for (int u4 = 0; u4 < 8; ++u4) {
                    const float4 c4 = __ldg(ys4 + u4);
                    v[u4 * 4 + 0] *= c4.x;
                    v[u4 * 4 + 1] *= c4.y;
                    v[u4 * 4 + 2] *= c4.z;
                    v[u4 * 4 + 3] *= c4.w;
                }
                float c4m[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) c4m[a] = ninf<float>();
#pragma unroll
                for (int u = 0; u < 32; ++u) c4m[u & 3] = fmaxf(c4m[u & 3], v[u]);
                const float cmax = fmaxf(fmaxf(c4m[0], c4m[1]), fmaxf(c4m[2], c4m[3])) * c1r;
                if (cmax > m) {
                    l *= ExpTraits<float>::bexp(m - cmax);
                    m = cmax;
                }
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int u = 0; u < 32; ++u) s4[u & 3] += ExpTraits<float>::bexp(fmaf(v[u], c1r, -m));
                l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
                continue;
            }
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4) {
                const float4 c4 = __ldg(ys4 + u4);
                const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int u = u4 * 4 + k;
                    const float raw = v[u] * cs[k];
                    float sc;
                    if (METRIC == kLinear && !EXP) {
                        sc = raw * c1r;
                    } else {
                        const int64_t j = j0 + u;
                        float dot = raw * xs;
                        if (METRIC != kLinear && masked && p.same && j == row) dot = xn;  // |x - x|^2 = 0 exactly
                        const float yn = (METRIC != kLinear && j < p.M) ? __ldg(p.yn + j) : 0.f;
                        sc = score2<METRIC, EXP>(dot, xn, yn, p.scale, p.neg_gamma_log2);
                    }
                    if (masked) {
                        const int64_t j = j0 + u;
                        if (j >= p.M || (p.exclude_self && j == row) || !pair_in(p.sc.pm, p.sc.band, row, j))
                            sc = ninf<float>();
                    }
                    v[u] = sc;
                }
            }
            float c4m[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) c4m[a] = ninf<float>();
#pragma unroll
            for (int u = 0; u < 32; ++u) c4m[u & 3] = fmaxf(c4m[u & 3], v[u]);
            const float cmax = fmaxf(fmaxf(c4m[0], c4m[1]), fmaxf(c4m[2], c4m[3]));
            if (cmax != ninf<float>()) {
                if (cmax > m) {
                    l *= ExpTraits<float>::bexp(m - cmax);
                    m = cmax;
                }
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int u = 0; u < 32; ++u) s4[u & 3] += ExpTraits<float>::bexp(v[u] - m);
                l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
            }
        }
        if (ok && rb_cur >= 0) flush();
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------------------------
// Forward over the upper triangle, for X = Y with a linear score without exp and no pair mask (the
// InfoNCE row). The score matrix is symmetric, so each tile (I, J), J >= I, of 128 x 128 is evaluated
// once for the rows of both blocks. The terms are taken against one fixed offset, e_ij = 2^(s2_ij - M)
// with M = |scale| log2(e) max|x|^2 >= every s2 (Cauchy-Schwarz), which makes them symmetric as well:
// a tile's row sums belong to the rows of I and its column sums to the rows of J. When 2 M <= 120 every
// term is a normal fp32 number, so nothing underflows and no running maximum is needed; otherwise the
// kernel sets the fallback flag and returns, and lse_fwd_tc runs the full sweep with running maxima.
// A diagonal tile (J = I) covers both orders of its pairs and counts for its rows only. Each CTA walks a
// contiguous range of the triangle's tiles numbered row-block major; it writes one row partial per row
// block of its range and one column partial per off-diagonal tile, and lse_fwd_tc (merge mode) adds
// them in a fixed order.
// ------------------------------------------------------------------------------------------------
constexpr float kSymSpan = 120.f;  // 2 M: the widest range of exponents the terms may span
constexpr int kSymCap = 96;        // row blocks: the column partials grow with their square
constexpr int kTrW = 36;           // the epilogue warps' transpose buffers: 32 rows x 32 columns, padded
constexpr int kStY = 3;            // column stages (the transposes take the fourth's room)
constexpr size_t kSmemS = (size_t)kPairF * (1 + kStY) + 256 + 1024 + (size_t)kEpi * 32 * kTrW * 4;
static_assert(kSmemS <= 232448, "dynamic shared memory per CTA");

struct LseSymParams {
    int64_t N;
    int RB;       // row blocks of 128
    int64_t T;    // tiles of the triangle: RB (RB + 1) / 2
    int G;        // CTAs
    int exclude_self;
    float scale;
    const float* xs;    // 2^-e of each point (padded to whole row blocks, zeros past N)
    const float* xn;    // |x_i|^2 (zeros past N)
    float* prow;        // [RB + G][128][4 column parts]: row sums, slot row block + CTA
    float* pcol;        // [T][128][4 row quarters]: column sums of each off-diagonal tile
    int* sym;           // [2]: 1 if the sweep fell back (lse_fwd_tc sweeps), 0 if done; M as float bits
    int* err;
};

// M (base 2) from the largest |x|^2, the same value in every CTA and in the merge.
__device__ float sym_offset(const float* __restrict__ xn, int64_t N, float scale, float* red) {
    float w[16];  // sixteen independent loads in flight per thread (the array sits in L2)
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = 0.f;
    for (int64_t r0 = threadIdx.x; r0 < N; r0 += 16 * (int64_t)blockDim.x) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int64_t r = r0 + (int64_t)k * blockDim.x;
            if (r < N) w[k] = fmaxf(w[k], __ldg(xn + r));
        }
    }
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) v = fmaxf(v, w[k]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    __syncthreads();
    return fabsf(scale) * 1.4426950408889634f * m;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    lse_fwd_sym_tc(const __grid_constant__ CUtensorMap mXh, const __grid_constant__ CUtensorMap mXl,
                   const LseSymParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_base1024(smem_raw);
    unsigned char* sA = sm;                     // [hi 128 rows | lo 128 rows]
    unsigned char* sB = sm + kPairF;            // stage s at sB + s * kPairF: [hi 128 points | lo 128 points]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + (size_t)kPairF * (1 + kStY));
    uint64_t* a_full = bars + 0;
    uint64_t* a_empty = bars + 1;
    uint64_t* b_full = bars + 2;                 // [kStY]
    uint64_t* b_empty = b_full + kStY;           // [kStY]
    uint64_t* acc_full = b_empty + kStY;         // [2]
    uint64_t* acc_empty = acc_full + 2;          // [2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    float* red = reinterpret_cast<float*>(tslot + 2);                 // [18] block maxima (barrier area: 176 B)
    float* trb = reinterpret_cast<float*>(sm + (size_t)kPairF * (1 + kStY) + 256);  // [kEpi][32][kTrW]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t_begin = range_start(p.T, p.G, blockIdx.x), t_end = range_start(p.T, p.G, blockIdx.x + 1);

    if (threadIdx.x == 0) {
        prefetch_map(&mXh);
        prefetch_map(&mXl);
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int s = 0; s < kStY; ++s) {
            mbar_init(b_full + s, 1);
            mbar_init(b_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, kEpi);  // one arrival per epilogue warp
        }
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    griddep_wait();
    griddep_launch();
    const float M = sym_offset(p.xn, p.N, p.scale, red);
    const bool bounded = 2.f * M <= kSymSpan;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        p.sym[0] = bounded ? 0 : 1;
        p.sym[1] = __float_as_int(M);
    }

    if (!bounded) {
        // the full sweep runs instead
    } else if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer: row block I and column block J of each tile
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            SymCursor cur(t_begin, p.RB);
            for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next()) {
                const int64_t i = t - t_begin;
                if (cur.I != rb_cur) {
                    if (a_uses > 0) ok = mbar_wait(a_empty, (a_uses - 1) & 1, p.err, 91);
                    if (!ok) break;
                    mbar_expect_tx(a_full, kPairF);
                    tma_load_2d(sA, &mXh, 0, cur.I * kBM, a_full);
                    tma_load_2d(sA + kHalfTile, &mXl, 0, cur.I * kBM, a_full);
                    ++a_uses;
                    rb_cur = cur.I;
                }
                const int s = (int)(i % kStY), r = (int)(i / kStY);
                if (r >= 1) ok = mbar_wait(b_empty + s, (r - 1) & 1, p.err, 92);
                if (!ok) break;
                unsigned char* dst = sB + (size_t)s * kPairF;
                mbar_expect_tx(b_full + s, kPairF);
                tma_load_2d(dst, &mXh, 0, cur.J * kBN, b_full + s);
                tma_load_2d(dst + kHalfTile, &mXl, 0, cur.J * kBN, b_full + s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer (as lse_fwd_tc)
            constexpr uint32_t id256 = idesc_f16(kBM, 2 * kBN, false);
            constexpr uint32_t id128 = idesc_f16(kBM, kBN, false);
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            SymCursor cur(t_begin, p.RB);
            for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next()) {
                const int64_t i = t - t_begin;
                if (cur.I != rb_cur) {
                    if (a_uses > 0) mma_commit(a_empty);
                    ok = mbar_wait(a_full, a_uses & 1, p.err, 93);
                    if (!ok) break;
                    ++a_uses;
                    rb_cur = cur.I;
                }
                const int s = (int)(i % kStY), r = (int)(i / kStY), b = (int)(i & 1), rr = (int)(i >> 1);
                ok = mbar_wait(b_full + s, r & 1, p.err, 94);
                if (ok && rr >= 1) ok = mbar_wait(acc_empty + b, (rr - 1) & 1, p.err, 95);
                if (!ok) break;
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * 256);
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB + (size_t)s * kPairF);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ko = (uint32_t)(ks * 32);
                    mma_f16(d, desc_sw128(a0 + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), id256, ks > 0 ? 1u : 0u);
                    mma_f16(d + 128, desc_sw128(a0 + kHalfTile + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), id128,
                            1u);
                }
                mma_commit(b_empty + s);
                mma_commit(acc_full + b);
            }
        }
    } else {  // ---------------- epilogue: one row per thread, 32 of the tile's columns per warp
        constexpr float kL2E = 1.4426950408889634f;
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int sub = (warp - 2) >> 2;        // columns [32 sub, 32 sub + 32) of each tile
        const int lr = q * 32 + lane;           // row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(sub * 32);
        float* tr = trb + (size_t)(warp - 2) * 32 * kTrW;
        int rb_cur = -1;
        float rs = 0.f, c1r = 0.f;
        bool ok = true;
        auto flush = [&]() {
            p.prow[((size_t)(rb_cur + blockIdx.x) * kBM + lr) * 4 + sub] = rs;
        };
        SymCursor cur(t_begin, p.RB);
        for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next()) {
            const int64_t i = t - t_begin;
            const int I = cur.I, J = cur.J;
            const int64_t row = (int64_t)I * kBM + lr;
            if (I != rb_cur) {
                if (rb_cur >= 0) flush();
                rs = 0.f;
                rb_cur = I;
                c1r = p.scale * kL2E * __ldg(p.xs + row);  // 0 for padding rows
            }
            const int b = (int)(i & 1), rr = (int)(i >> 1);
            ok = mbar_wait_warp(acc_full + b, rr & 1, p.err, 96);
            if (!ok) break;
            fence_after_sync();
            float e[32];  // hi*hi + (hi*lo + lo*hi), then the terms
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                float t0[16], t1[16];
                tmem_ld16x2(lane_base + (uint32_t)(b * 256 + hlf * 16), lane_base + (uint32_t)(b * 256 + 128 + hlf * 16),
                            t0, t1);
#pragma unroll
                for (int u = 0; u < 16; ++u) e[hlf * 16 + u] = t0[u] + t1[u];
            }
            fence_before_sync();
            mbar_arrive_warp(acc_empty + b);  // the values are in registers: the MMA may reuse the buffer
            const int64_t j0 = (int64_t)J * kBN + sub * 32;
            const float4* ys4 = reinterpret_cast<const float4*>(p.xs + j0);  // padded: 32 readable entries
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4) {
                const float4 c4 = __ldg(ys4 + u4);
                e[u4 * 4 + 0] = ExpTraits<float>::bexp(fmaf(e[u4 * 4 + 0] * c4.x, c1r, -M));
                e[u4 * 4 + 1] = ExpTraits<float>::bexp(fmaf(e[u4 * 4 + 1] * c4.y, c1r, -M));
                e[u4 * 4 + 2] = ExpTraits<float>::bexp(fmaf(e[u4 * 4 + 2] * c4.z, c1r, -M));
                e[u4 * 4 + 3] = ExpTraits<float>::bexp(fmaf(e[u4 * 4 + 3] * c4.w, c1r, -M));
            }
            // columns past N, and the pair (i, i) when it is excluded, add nothing (rows past N occur in the
            // last diagonal tile only, whose row sums are not merged)
            const bool diag = I == J;
            const int64_t lim = p.N - j0, self = (diag && p.exclude_self) ? row - j0 : -1;
            if (__any_sync(0xffffffffu, lim < 32 || (self >= 0 && self < 32))) {
#pragma unroll
                for (int u = 0; u < 32; ++u) e[u] = (u >= lim || u == self) ? 0.f : e[u];
            }
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int u = 0; u < 32; ++u) s4[u & 3] += e[u];
            rs += (s4[0] + s4[1]) + (s4[2] + s4[3]);
            if (!diag) {
                // column sums over the warp's 32 rows through shared memory (row stride 36 floats: the
                // 16-byte stores of eight lanes and the column reads of 32 lanes hit distinct banks)
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<float4*>(tr + lane * kTrW + 4 * k) =
                        make_float4(e[4 * k], e[4 * k + 1], e[4 * k + 2], e[4 * k + 3]);
                __syncwarp();
                float c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int r = 0; r < 32; ++r) c4[r & 3] += tr[r * kTrW + lane];
                p.pcol[((size_t)t * kBM + sub * 32 + lane) * 4 + q] = (c4[0] + c4[1]) + (c4[2] + c4[3]);
            }
        }
        if (ok && rb_cur >= 0) flush();
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------------------------
// Symmetric backward (X = Y = z, no row/column parameters): z.grad_k = sum_j kappa_kj z_j
// - [distance metric] z_k sum_j kappa_kj, with kappa_kj the coefficient of z_j in d/dz_k of
// g_k lse_k + g_j lse_j: G = g_k P_kj + g_j P_jk (P_kj = exp(S_kj - lse_k)), H = G (times S with
// exp), E = H * scale, kappa = E (linear), -2E (sqeuclidean), 2 gamma E base (rbf). Each pair is
// evaluated once, for both sides of the pair at the same time.
//
// Per 64-column tile: S = Zrows Ztile^T into TMEM; the epilogue turns S into kappa, scales each row's
// kappa by a power of two (agreed by the four warps that share the row), splits it into fp16 hi/lo and
// stores it back into TMEM, two values per column; then dZ = kappa_hi [Zh | Zl] + kappa_lo Zh with
// kappa as the A operand read from TMEM. The B operand of dZ is the same point-major tile as for S,
// read MN-major (64 features contiguous per point), so one 16 KB tile per 64 columns feeds both
// contractions. Each tile's dZ (128 x 64) lands in a TMEM block of its own and the epilogue adds it,
// unscaled, into a per-row register accumulator: the tensor core's accumulation never spans more
// than one tile, and the rows' sums are two-level like everywhere else. At the end of the CTA's
// share of a row block the accumulator is written as a partial; the last CTA to finish the row block
// adds the partials of each row in CTA order.
//
// Order of the MMAs: S runs two tiles ahead of dZ (three S buffers in TMEM), so the S of tile i+1 is
// ready when the epilogue finishes tile i.
// ------------------------------------------------------------------------------------------------
constexpr int kBNb = 64;                   // columns per backward tile
constexpr int kTileB = kBNb * kRowBytes;   // 64 points of hi (or lo): 8 KB
constexpr int kStageB = 2 * kTileB;        // [hi 64 points | lo 64 points]: one 128-row operand, 16 KB
constexpr int kStagesS = 4;                // a stage lives from its S MMA until its dZ MMA
constexpr int kSBuf = 3;                   // S / kappa buffers in TMEM (128 columns each)
constexpr uint32_t kDZCol = kSBuf * 128;   // the dZ buffer (128 columns)
constexpr int kPartsB = kEpi / 4;          // epilogue warps per lane quarter, each owning 16 columns
constexpr int kColsB = kBNb / kPartsB;     // 16: one K step of the dZ MMA
constexpr int kPartRowsB = 64 + kPartsB;   // rows of one partial: 64 dZ features + one kappa sum per part
// shared memory: row block A (hi, lo: 32 KB), kStagesS operand stages, their (lse, g, 2^-e) column stats,
// the per-quarter exchange of row maxima (two tile parities), barriers, alignment slack
constexpr size_t kSmemB = (size_t)kPairF + (size_t)kStageB * kStagesS + (size_t)kStagesS * kBNb * 16 +
                          2 * 4 * kPartsB * 32 * 4 + 512 + 1024;
static_assert(kSmemB <= 232448, "dynamic shared memory per CTA");
static_assert(kColsB == 16, "one dZ K step per epilogue warp");

struct LseBwdTcParams {
    int64_t N;
    int64_t T;
    int CT, G, smax;
    int metric, apply_exp, exclude_self;
    float scale, neg_gamma_log2, two_gamma;
    const float* zn;      // |z_k|^2
    const float4* stat;   // [ceil(N/64)*64]: (lse_j log2 e, g_j, 2^-e_j, scale 2^-e_j), padding (+inf, 0, 0, 0)
    float* part;          // [G][smax][kPartRowsB][128]: dZ features, then each part's sum of kappa, row-minor
    int* cnt;             // [RB] CTAs done with each row block (zeroed by the pre-pass)
    const float* z;       // [N][64] the points (distance metrics subtract z_k sum_j kappa_kj)
    float* grad;          // [N][64] output: z.grad
    const int* gmax;      // linear score without exp: (max|z|, max|g|) as float bits
    int* err;
};

// Linear score without exp: z carries one power of two e (max|z| 2^e in [2^14, 2^15)), and kappa one
// power of two E fixed from the bound |kappa_kj| = |scale| |g_k P_kj + g_j P_jk| <= 2 |scale| max|g|
// (P <= 1 off the diagonal), so both are constants of the whole sweep.
__device__ __forceinline__ int lin_z_exp(const int* gm) { return f16_row_exponent(__int_as_float(__ldg(gm))); }
__device__ __forceinline__ int lin_kappa_exp(const int* gm, float scale) {
    return f16_row_exponent(2.f * fabsf(scale) * __int_as_float(__ldg(gm + 1)));
}

// z.grad for features [16 fg, 16 fg + 16) of row lr of row block rb from the partials of every CTA that
// saw the row block, added in CTA order: dZ - [distance metric] z sum kappa.
__device__ __noinline__ void bwd_merge_row(const LseBwdTcParams& p, int rb, int lr, int fg) {
    const int64_t row = (int64_t)rb * kBM + lr;
    if (row >= p.N) return;
    const int64_t t0 = (int64_t)rb * p.CT;
    const int c_lo = cta_of_tile(p.T, p.G, t0), c_hi = cta_of_tile(p.T, p.G, t0 + p.CT - 1);
    float acc[16], k0 = 0.f;
#pragma unroll
    for (int f = 0; f < 16; ++f) acc[f] = 0.f;
    for (int c = c_lo; c <= c_hi; ++c) {
        const int seg = rb - rb_of_tile(range_start(p.T, p.G, c), p.CT);
        const float* o = p.part + (size_t)(c * p.smax + seg) * kPartRowsB * kBM + lr;
#pragma unroll
        for (int f = 0; f < 16; ++f) acc[f] += __ldcg(o + (size_t)(fg * 16 + f) * kBM);
        if (p.metric != kLinear) {
#pragma unroll
            for (int qq = 0; qq < kPartsB; ++qq) k0 += __ldcg(o + (size_t)(64 + qq) * kBM);
        }
    }
    float4* g4 = reinterpret_cast<float4*>(p.grad + row * 64 + fg * 16);
    if (p.metric == kLinear) {
#pragma unroll
        for (int f4 = 0; f4 < 4; ++f4) g4[f4] = make_float4(acc[4 * f4], acc[4 * f4 + 1], acc[4 * f4 + 2], acc[4 * f4 + 3]);
    } else {
        const float4* z4 = reinterpret_cast<const float4*>(p.z + row * 64 + fg * 16);
#pragma unroll
        for (int f4 = 0; f4 < 4; ++f4) {
            const float4 zz = z4[f4];
            g4[f4] = make_float4(acc[4 * f4] - zz.x * k0, acc[4 * f4 + 1] - zz.y * k0, acc[4 * f4 + 2] - zz.z * k0,
                                 acc[4 * f4 + 3] - zz.w * k0);
        }
    }
}

template <int METRIC, bool EXP>
__global__ void __launch_bounds__(kTcThreads, 1)
    lse_bwd_sym_tc(const __grid_constant__ CUtensorMap mAh, const __grid_constant__ CUtensorMap mAl,
                   const __grid_constant__ CUtensorMap mBh, const __grid_constant__ CUtensorMap mBl,
                   const LseBwdTcParams p) {
    constexpr float kL2E = 1.4426950408889634f;
    extern __shared__ unsigned char smem_raw[];
    // aligned through an integer address (generic loads): derived from the array itself, this kernel's
    // register allocation spills 150-200 bytes
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = sm;                                        // row block: [hi 128 rows | lo 128 rows]
    unsigned char* sB = sm + kPairF;                               // stage s: [hi 64 points | lo 64 points]
    float4* sStat = reinterpret_cast<float4*>(sB + (size_t)kStageB * kStagesS);  // [stage][64]
    float* sMax = reinterpret_cast<float*>(sStat + kStagesS * kBNb);             // [parity][quarter][part][lane]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sMax + 2 * 4 * kPartsB * 32);
    uint64_t* a_full = bars + 0;
    uint64_t* a_empty = bars + 1;
    uint64_t* bs_full = bars + 2;                // [kStagesS]
    uint64_t* bs_empty = bs_full + kStagesS;     // [kStagesS]
    uint64_t* s_full = bs_empty + kStagesS;      // [kSBuf]
    uint64_t* w_full = s_full + kSBuf;           // [kSBuf]
    uint64_t* dz_full = w_full + kSBuf;
    uint64_t* dz_empty = dz_full + 1;
    uint64_t* xch = dz_empty + 1;                // [quarter][parity]: the row-maximum exchange
    uint64_t* fl_bar = xch + 8;                  // the epilogue wrote its partials of a row block
    uint64_t* dec_bar = fl_bar + 1;              // the CTA knows whether it merges that row block
    uint32_t* tslot = reinterpret_cast<uint32_t*>(dec_bar + 1);
    volatile int* sflag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t_begin = range_start(p.T, p.G, blockIdx.x), t_end = range_start(p.T, p.G, blockIdx.x + 1);
    const int64_t n = t_end - t_begin;

    if (threadIdx.x == 0) {
        prefetch_map(&mAh);
        prefetch_map(&mAl);
        prefetch_map(&mBh);
        prefetch_map(&mBl);
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int s = 0; s < kStagesS; ++s) {
            mbar_init(bs_full + s, 1);
            mbar_init(bs_empty + s, 1);
        }
        for (int b = 0; b < kSBuf; ++b) {
            mbar_init(s_full + b, 1);
            mbar_init(w_full + b, 32 * kEpi);
        }
        mbar_init(dz_full, 1);
        mbar_init(dz_empty, 32 * kEpi);
        for (int x = 0; x < 8; ++x) mbar_init(xch + x, 32 * kPartsB);
        mbar_init(fl_bar, 32 * kEpi);
        mbar_init(dec_bar, 1);
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    griddep_wait();
    griddep_launch();
    const uint32_t tDZ = tmem + kDZCol;

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer: operand stages in tile order
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            TileCursor cur(t_begin, p.CT);
            for (int64_t i = 0; i < n && ok; ++i, cur.next()) {
                const int rb = cur.rb, ct = cur.ct;
                if (rb != rb_cur) {
                    if (a_uses > 0) ok = mbar_wait(a_empty, (a_uses - 1) & 1, p.err, 21);
                    if (!ok) break;
                    mbar_expect_tx(a_full, kPairF);
                    tma_load_2d(sA, &mAh, 0, rb * kBM, a_full);
                    tma_load_2d(sA + kHalfTile, &mAl, 0, rb * kBM, a_full);
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStagesS), r = (int)(i / kStagesS);
                if (r >= 1) ok = mbar_wait(bs_empty + s, (r - 1) & 1, p.err, 22);
                if (!ok) break;
                unsigned char* dst = sB + (size_t)s * kStageB;
                mbar_expect_tx(bs_full + s, kStageB + kBNb * 16);
                tma_load_2d(dst, &mBh, 0, ct * kBNb, bs_full + s);
                tma_load_2d(dst + kTileB, &mBl, 0, ct * kBNb, bs_full + s);
                bulk_load(sStat + s * kBNb, p.stat + (size_t)ct * kBNb, kBNb * 16, bs_full + s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            constexpr uint32_t idS2 = idesc_f16(kBM, 2 * kBNb, false);  // Zh [Zth; Ztl]: N 128
            constexpr uint32_t idS = idesc_f16(kBM, kBNb, false);       // Zl Zth: N 64
            constexpr uint32_t idZ2 = idesc_f16(kBM, 128, true);        // kappa_hi [Zh | Zl] (MN-major): N 128
            constexpr uint32_t idZ = idesc_f16(kBM, 64, true);          // kappa_lo Zh (MN-major): N 64
            int a_uses = 0, rb_cur = -1;
            bool ok = true;
            TileCursor cur(t_begin, p.CT);
            // S for tile j into S buffer j % kSBuf (its previous kappa was read by dZ(j - kSBuf), issued earlier)
            auto issue_s = [&](int64_t j) -> bool {
                const int rb = cur.rb;
                cur.next();
                if (rb != rb_cur) {
                    if (a_uses > 0) mma_commit(a_empty);  // the old A is free once its MMAs finish
                    if (!mbar_wait(a_full, a_uses & 1, p.err, 23)) return false;
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(j % kStagesS), r = (int)(j / kStagesS), b = (int)(j % kSBuf);
                if (!mbar_wait(bs_full + s, r & 1, p.err, 24)) return false;
                fence_after_sync();
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB + (size_t)s * kStageB);
                const uint32_t d = tmem + (uint32_t)(b * 128);
                // per 16 features: Zh [Zth; Ztl] (hi*hi into columns 0..63, hi*lo into 64..127), then Zl Zth
                // into 64..127
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ko = (uint32_t)(ks * 32);
                    mma_f16(d, desc_sw128(a0 + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), idS2, ks > 0 ? 1u : 0u);
                    mma_f16(d + 64, desc_sw128(a0 + kHalfTile + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), idS, 1u);
                }
                mma_commit(s_full + b);
                return true;
            };
            // dZ for tile i (kappa in TMEM): once its epilogue is done and has drained the previous dZ
            auto issue_dz = [&](int64_t i) -> bool {
                const int b = (int)(i % kSBuf), s = (int)(i % kStagesS);
                if (!mbar_wait(w_full + b, (uint32_t)((i / kSBuf) & 1), p.err, 25)) return false;
                if (i >= 1 && !mbar_wait(dz_empty, (uint32_t)((i - 1) & 1), p.err, 26)) return false;
                fence_after_sync();
                const uint32_t b0 = smem_u32(sB + (size_t)s * kStageB);
                const uint32_t kh = tmem + (uint32_t)(b * 128), kl = kh + 32;  // packed kappa_hi, kappa_lo
                // per 16 points (one epilogue part): the stage read MN-major, rows of 16 points, hi and lo
                // feature blocks kTileB apart
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t bo = b0 + (uint32_t)(ks * 16 * kRowBytes);
                    mma_f16_ta(tDZ, kh + (uint32_t)(ks * 8), desc_sw128(bo, kTileB, 1024), idZ2, ks > 0 ? 1u : 0u);
                    mma_f16_ta(tDZ + 64, kl + (uint32_t)(ks * 8), desc_sw128(bo, kTileB, 1024), idZ, 1u);
                }
                mma_commit(bs_empty + s);  // the stage fed both S and dZ
                mma_commit(dz_full);
                return true;
            };
            // S(i + 2) goes in before the wait for tile i's kappa: its buffer last held kappa(i - 1), read by
            // dZ(i - 1), already issued; so the tensor pipe works on it while the epilogue finishes tile i
            for (int64_t j = 0; j < n && j < 2 && ok; ++j) ok = issue_s(j);
            for (int64_t i = 0; i < n && ok; ++i) {
                if (i + 2 < n) ok = issue_s(i + 2);
                if (ok) ok = issue_dz(i);
            }
        }
    } else {
        // ---------------- epilogue: four warps per TMEM lane quarter; part p owns tile columns
        // [16 p, 16 p + 16) (one dZ K step) and dZ features [16 p, 16 p + 16)
        const int q = warp & 3;
        const int part = (warp - 2) >> 2;
        const int lr = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int N32 = (int)p.N;
        int seg = 0;
        float K0 = 0.f, lse2k = 0.f, gk = 0.f, zn_k = 0.f, rs_k = 0.f, rsl = 0.f;
        float dacc[kColsB];
#pragma unroll
        for (int f = 0; f < kColsB; ++f) dacc[f] = 0.f;
        bool ok = true;
        // add this part of tile j's dZ block, scaled back by inv, into the row accumulator
        auto drain = [&](int64_t j, float inv) -> bool {
            if (!mbar_wait(dz_full, (uint32_t)(j & 1), p.err, 27)) return false;
            fence_after_sync();
            float v[kColsB], w[kColsB];
            tmem_ld16x2(tDZ + lane_off + (uint32_t)(part * kColsB), tDZ + lane_off + (uint32_t)(64 + part * kColsB), v, w);
#pragma unroll
            for (int u = 0; u < kColsB; ++u) dacc[u] += (v[u] + w[u]) * inv;
            fence_before_sync();
            mbar_arrive(dz_empty);
            return true;
        };
        int rb_cur = -1, row = 0;
        const int etid = threadIdx.x - 64;  // 0 .. 32 kEpi - 1
        // Write this thread's partial of row block rb_cur. The CTA that completes the row block (the last
        // of the CTAs whose tile ranges meet it to count itself in) merges it into z.grad.
        auto write_partial = [&]() {
            float* o = p.part + (size_t)(blockIdx.x * p.smax + seg) * kPartRowsB * kBM;
#pragma unroll
            for (int f = 0; f < kColsB; ++f) o[(size_t)(part * kColsB + f) * kBM + lr] = dacc[f];
            o[(size_t)(64 + part) * kBM + lr] = K0;
            __threadfence();
            mbar_arrive(fl_bar);
            if (etid == 0) {
                int last = 0;
                if (mbar_wait(fl_bar, (uint32_t)(seg & 1), p.err, 33)) {
                    const int64_t t0 = (int64_t)rb_cur * p.CT;
                    const int need = cta_of_tile(p.T, p.G, t0 + p.CT - 1) - cta_of_tile(p.T, p.G, t0) + 1;
                    last = atomicAdd(p.cnt + rb_cur, 1) + 1 == need;
                    __threadfence();
                }
                *sflag = last;
                mbar_arrive(dec_bar);
            }
            if (mbar_wait(dec_bar, (uint32_t)(seg & 1), p.err, 34) && *sflag) bwd_merge_row(p, rb_cur, etid % kBM, etid / kBM);
            ++seg;
        };
        int64_t pending = -1;
        float pend_inv = 0.f;
        TileCursor cur(t_begin, p.CT);
        for (int64_t i = 0; i < n && ok; ++i, cur.next()) {
            const int rb = cur.rb, ct = cur.ct;
            if (rb != rb_cur) {
                if (pending >= 0) {
                    ok = drain(pending, pend_inv);
                    pending = -1;
                    if (!ok) break;
                }
                if (rb_cur >= 0) write_partial();
                rb_cur = rb;
                row = rb * kBM + lr;
                K0 = 0.f;
#pragma unroll
                for (int f = 0; f < kColsB; ++f) dacc[f] = 0.f;
                const bool live = row < N32;
                const float4 st = live ? p.stat[row] : make_float4(__int_as_float(0x7f800000), 0.f, 0.f, 0.f);
                lse2k = st.x;
                gk = st.y;
                rs_k = st.z;
                rsl = rs_k * p.scale * kL2E;
                zn_k = (METRIC != kLinear && live) ? p.zn[row] : 0.f;
            }
            const int b = (int)(i % kSBuf), s = (int)(i % kStagesS);
            ok = mbar_wait(s_full + b, (uint32_t)((i / kSBuf) & 1), p.err, 28) &&
                 mbar_wait(bs_full + s, (uint32_t)((i / kStagesS) & 1), p.err, 31);  // the tile's column stats
            if (!ok) break;
            fence_after_sync();
            const int j0 = ct * kBNb + part * kColsB;
            const int lim = N32 - j0;                        // columns u >= lim are padding
            const int self = row - j0;                       // column u == self is the pair (row, row)
            const int dead_self = p.exclude_self ? self : -1;
            const float4* st = sStat + s * kBNb + part * kColsB;
            const uint32_t col = (uint32_t)(b * 128 + part * kColsB);
            float v[kColsB], w[kColsB];
            tmem_ld16x2(tmem + lane_off + col, tmem + lane_off + col + 64, v, w);  // hi*hi, hi*lo + lo*hi
            float ksum = 0.f, pm = 0.f;
            // columns that need care in this warp: padding past N, or the pair (row, row)
            const bool edge = lim < kColsB || (self >= 0 && self < kColsB && (p.exclude_self || METRIC != kLinear));
            if (METRIC == kLinear && !EXP && !__any_sync(0xffffffffu, edge)) {
                // common case: s2 = (x.y 2^(e_k+e_j)) 2^-e_j 2^-e_k scale log2(e); kappa 2^-e_j = G scale 2^-e_j
#pragma unroll
                for (int u = 0; u < kColsB; ++u) {
                    const float4 sj = st[u];
                    const float s2 = (v[u] + w[u]) * sj.z * rsl;
                    const float G = gk * ExpTraits<float>::bexp(s2 - lse2k) + sj.y * ExpTraits<float>::bexp(s2 - sj.x);
                    const float kp = G * sj.w;
                    v[u] = kp;
                    pm = fmaxf(pm, fabsf(kp));
                }
            } else {
#pragma unroll
            for (int u = 0; u < kColsB; ++u) {
                const float4 sj = st[u];                     // (lse_j log2 e, g_j, 2^-e_j, scale 2^-e_j)
                float dot = (v[u] + w[u]) * sj.z * rs_k;
                if (METRIC != kLinear && u == self) dot = zn_k;  // |z - z|^2 = 0 exactly
                float base;
                if (METRIC == kLinear) {
                    base = dot;
                } else {
                    const float d2 = fmaxf(fmaf(-2.f, dot, zn_k + __ldg(p.zn + (u < lim ? j0 + u : 0))), 0.f);
                    base = METRIC == kRbf ? ExpTraits<float>::bexp(p.neg_gamma_log2 * d2) : d2;
                }
                const float tt = p.scale * base;
                const float S = EXP ? ExpTraits<float>::bexp(tt * kL2E) : tt;
                const float s2 = S * kL2E;
                const float G = gk * ExpTraits<float>::bexp(s2 - lse2k) + sj.y * ExpTraits<float>::bexp(s2 - sj.x);
                const bool dead = u >= lim || u == dead_self;
                const float H = EXP ? G * S : G;
                const float E = H * p.scale;
                float kap = METRIC == kLinear ? E : (METRIC == kSqeuclidean ? -2.f * E : p.two_gamma * E * base);
                kap = dead ? 0.f : kap;
                ksum += kap;
                const float kp = kap * sj.z;                 // z_j = 2^-e_j (z_j 2^e_j): fold the column's scale
                v[u] = kp;
                pm = fmaxf(pm, fabsf(kp));
            }
            }
            K0 += ksum;
            // the row's largest |kappa 2^-e_j| over the tile: the four parts of the quarter exchange theirs
            const int par = (int)(i & 1);
            float* xm = sMax + (size_t)((par * 4 + q) * kPartsB) * 32;
            xm[part * 32 + lane] = pm;
            fence_before_sync();
            mbar_arrive(xch + q * 2 + par);
            ok = mbar_wait(xch + q * 2 + par, (uint32_t)((i >> 1) & 1), p.err, 32);
            if (!ok) break;
            fence_after_sync();
            float mx = xm[lane];
#pragma unroll
            for (int pp = 1; pp < kPartsB; ++pp) mx = fmaxf(mx, xm[pp * 32 + lane]);
            const int e = f16_row_exponent(mx);
            const float f = pow2i(e);
            uint32_t hw[kColsB / 2], lw[kColsB / 2];
#pragma unroll
            for (int k = 0; k < kColsB / 2; ++k) {
                const float a = v[2 * k] * f, c = v[2 * k + 1] * f;
                const __half2 h = __floats2half2_rn(a, c);
                const float2 hf = __half22float2(h);
                hw[k] = *reinterpret_cast<const uint32_t*>(&h);
                lw[k] = pack_f16x2(a - hf.x, c - hf.y);
            }
            // kappa_hi of points [16 part, 16 part + 16) in columns b*128 + 8 part .. +8, kappa_lo 32 further
            tmem_st8(tmem + lane_off + (uint32_t)(b * 128 + part * 8), hw);
            tmem_st8(tmem + lane_off + (uint32_t)(b * 128 + 32 + part * 8), lw);
            tmem_st_wait();
            fence_before_sync();
            mbar_arrive(w_full + b);
            if (pending >= 0) {
                ok = drain(pending, pend_inv);
                if (!ok) break;
            }
            pending = i;
            pend_inv = pow2i(-e);
        }
        if (ok && pending >= 0) ok = drain(pending, pend_inv);
        if (ok && rb_cur >= 0) write_partial();
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------------------------
// Symmetric backward, linear score without exp: the epilogue is two groups of eight warps (two per TMEM
// lane quarter) that take alternate tiles, each group with an S buffer and a dZ accumulator of its own
// in TMEM. One group's TMEM loads, stores and drains then overlap the other group's arithmetic, and the
// tensor core runs the S and dZ MMAs of the two groups back to back. A warp covers 32 of the tile's 64
// columns (two K steps of the dZ MMA) and 32 of the 64 dZ features. Both groups flush a partial for every
// row block of the CTA's range, in order (zeros where a group had no tile), so the row-block completion
// protocol sees both; the merge adds the two groups' slices.
// ------------------------------------------------------------------------------------------------
constexpr int kGrpW = kEpi / 2;             // warps per epilogue group
constexpr int kPartRowsL = 128;             // rows of one partial: 64 dZ features per group

// z.grad for features [16 fg, 16 fg + 16) of row lr of row block rb: both groups' slices of the partials
// of every CTA that saw the row block, added in CTA order.
__device__ __noinline__ void lin_merge_row(const LseBwdTcParams& p, int rb, int lr, int fg) {
    const int64_t row = (int64_t)rb * kBM + lr;
    if (row >= p.N) return;
    const int64_t t0 = (int64_t)rb * p.CT;
    const int c_lo = cta_of_tile(p.T, p.G, t0), c_hi = cta_of_tile(p.T, p.G, t0 + p.CT - 1);
    float acc[16];
#pragma unroll
    for (int f = 0; f < 16; ++f) acc[f] = 0.f;
    for (int c = c_lo; c <= c_hi; ++c) {
        const int seg = rb - rb_of_tile(range_start(p.T, p.G, c), p.CT);
        const float* o = p.part + (size_t)(c * p.smax + seg) * kPartRowsL * kBM + lr;
#pragma unroll
        for (int f = 0; f < 16; ++f)
            acc[f] += __ldcg(o + (size_t)(fg * 16 + f) * kBM) + __ldcg(o + (size_t)(64 + fg * 16 + f) * kBM);
    }
    float4* g4 = reinterpret_cast<float4*>(p.grad + row * 64 + fg * 16);
#pragma unroll
    for (int f4 = 0; f4 < 4; ++f4) g4[f4] = make_float4(acc[4 * f4], acc[4 * f4 + 1], acc[4 * f4 + 2], acc[4 * f4 + 3]);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    lse_bwd_lin_tc(const __grid_constant__ CUtensorMap mAh, const __grid_constant__ CUtensorMap mAl,
                   const __grid_constant__ CUtensorMap mBh, const __grid_constant__ CUtensorMap mBl,
                   const LseBwdTcParams p) {
    constexpr float kL2E = 1.4426950408889634f;
    extern __shared__ unsigned char smem_raw[];
    // aligned through an integer address (generic loads): derived from the array itself, this kernel
    // measured 2% slower, and so did explicit shared-memory loads of its stage statistics alone
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = sm;                                        // row block: [hi 128 rows | lo 128 rows]
    unsigned char* sB = sm + kPairF;                               // stage s: [hi 64 points | lo 64 points]
    float4* sStat = reinterpret_cast<float4*>(sB + (size_t)kStageB * kStagesS);  // [stage][64]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStat + kStagesS * kBNb);
    uint64_t* a_full = bars + 0;
    uint64_t* a_empty = bars + 1;
    uint64_t* bs_full = bars + 2;                // [kStagesS]
    uint64_t* bs_empty = bs_full + kStagesS;     // [kStagesS]
    uint64_t* s_full = bs_empty + kStagesS;      // [2] per group: S of its tile is in its buffer
    uint64_t* w_full = s_full + 2;               // [2] the group stored its tile's kappa
    uint64_t* dz_full = w_full + 2;              // [2] the group's dZ block is complete
    uint64_t* dz_empty = dz_full + 2;            // [2] the group read its dZ block
    uint64_t* fl_bar = dz_empty + 2;             // the epilogue wrote its partials of a row block
    uint64_t* dec_bar = fl_bar + 1;              // the CTA knows whether it merges that row block
    uint32_t* tslot = reinterpret_cast<uint32_t*>(dec_bar + 1);
    volatile int* sflag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t_begin = range_start(p.T, p.G, blockIdx.x), t_end = range_start(p.T, p.G, blockIdx.x + 1);
    const int64_t n = t_end - t_begin;

    if (threadIdx.x == 0) {
        prefetch_map(&mAh);
        prefetch_map(&mAl);
        prefetch_map(&mBh);
        prefetch_map(&mBl);
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int s = 0; s < kStagesS; ++s) {
            mbar_init(bs_full + s, 1);
            mbar_init(bs_empty + s, 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(s_full + g, 1);
            mbar_init(w_full + g, kGrpW);  // one arrival per warp of the group
            mbar_init(dz_full + g, 1);
            mbar_init(dz_empty + g, kGrpW);
        }
        mbar_init(fl_bar, kEpi);
        mbar_init(dec_bar, 1);
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    griddep_wait();
    griddep_launch();
    // group g: S buffer at column 128 g (hi*hi 0..63, hi*lo + lo*hi 64..127), dZ at 256 + 128 g
    auto tS = [&](int g) { return tmem + (uint32_t)(128 * g); };
    auto tD = [&](int g) { return tmem + (uint32_t)(256 + 128 * g); };

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer: operand stages in tile order
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            TileCursor cur(t_begin, p.CT);
            for (int64_t i = 0; i < n && ok; ++i, cur.next()) {
                const int rb = cur.rb, ct = cur.ct;
                if (rb != rb_cur) {
                    if (a_uses > 0) ok = mbar_wait(a_empty, (a_uses - 1) & 1, p.err, 61);
                    if (!ok) break;
                    mbar_expect_tx(a_full, kPairF);
                    tma_load_2d(sA, &mAh, 0, rb * kBM, a_full);
                    tma_load_2d(sA + kHalfTile, &mAl, 0, rb * kBM, a_full);
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStagesS), r = (int)(i / kStagesS);
                if (r >= 1) ok = mbar_wait(bs_empty + s, (r - 1) & 1, p.err, 62);
                if (!ok) break;
                unsigned char* dst = sB + (size_t)s * kStageB;
                mbar_expect_tx(bs_full + s, kStageB + kBNb * 16);
                tma_load_2d(dst, &mBh, 0, ct * kBNb, bs_full + s);
                tma_load_2d(dst + kTileB, &mBl, 0, ct * kBNb, bs_full + s);
                bulk_load(sStat + s * kBNb, p.stat + (size_t)ct * kBNb, kBNb * 16, bs_full + s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            constexpr uint32_t idS2 = idesc_f16(kBM, 2 * kBNb, false);  // Zh [Zth; Ztl]: N 128
            constexpr uint32_t idS = idesc_f16(kBM, kBNb, false);       // Zl Zth: N 64
            constexpr uint32_t idZ2 = idesc_f16(kBM, 128, true);        // kappa_hi [Zh | Zl] (MN-major): N 128
            constexpr uint32_t idZ = idesc_f16(kBM, 64, true);          // kappa_lo Zh (MN-major): N 64
            int a_uses = 0, rb_cur = -1;
            bool ok = true;
            TileCursor cur(t_begin, p.CT);
            // S of tile j into its group's buffer (whose kappa(j - 2) was read by dZ(j - 2), issued before)
            auto issue_s = [&](int64_t j) -> bool {
                const int rb = cur.rb;
                cur.next();
                if (rb != rb_cur) {
                    if (a_uses > 0) mma_commit(a_empty);  // the old A is free once its MMAs finish
                    if (!mbar_wait(a_full, a_uses & 1, p.err, 63)) return false;
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(j % kStagesS), r = (int)(j / kStagesS), g = (int)(j & 1);
                if (!mbar_wait(bs_full + s, r & 1, p.err, 64)) return false;
                fence_after_sync();
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB + (size_t)s * kStageB);
                const uint32_t d = tS(g);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ko = (uint32_t)(ks * 32);
                    mma_f16(d, desc_sw128(a0 + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), idS2, ks > 0 ? 1u : 0u);
                    mma_f16(d + 64, desc_sw128(a0 + kHalfTile + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), idS, 1u);
                }
                mma_commit(s_full + g);
                return true;
            };
            // dZ of tile i from its kappa (stored by its group over the hi*hi S columns, K step ks at 16 ks)
            auto issue_dz = [&](int64_t i) -> bool {
                const int g = (int)(i & 1), s = (int)(i % kStagesS);
                if (!mbar_wait(w_full + g, (uint32_t)((i >> 1) & 1), p.err, 65)) return false;
                if (i >= 2 && !mbar_wait(dz_empty + g, (uint32_t)(((i >> 1) - 1) & 1), p.err, 66)) return false;
                fence_after_sync();
                const uint32_t b0 = smem_u32(sB + (size_t)s * kStageB);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t bo = b0 + (uint32_t)(ks * 16 * kRowBytes);
                    const uint32_t kh = tS(g) + (uint32_t)(ks * 16), kl = kh + 8;
                    mma_f16_ta(tD(g), kh, desc_sw128(bo, kTileB, 1024), idZ2, ks > 0 ? 1u : 0u);
                    mma_f16_ta(tD(g) + 64, kl, desc_sw128(bo, kTileB, 1024), idZ, 1u);
                }
                mma_commit(bs_empty + s);  // the stage fed both S and dZ
                mma_commit(dz_full + g);
                return true;
            };
            for (int64_t j = 0; j < n && j < 2 && ok; ++j) ok = issue_s(j);
            for (int64_t i = 0; i < n && ok; ++i) {
                ok = issue_dz(i);
                if (ok && i + 2 < n) ok = issue_s(i + 2);
            }
        }
    } else {
        // ---------------- epilogue: group grp takes the tiles i with i % 2 == grp; within it, half h of a lane
        // quarter owns tile columns [32 h, 32 h + 32) (dZ K steps 2h, 2h + 1) and dZ features [32 h, 32 h + 32)
        const int etid = threadIdx.x - 64;  // 0 .. 32 kEpi - 1
        const int grp = etid >> 8;
        const int q = warp & 3;
        const int half = ((warp - 2) >> 2) & 1;
        const int lr = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int N32 = (int)p.N;
        const int ez = lin_z_exp(p.gmax), E = lin_kappa_exp(p.gmax, p.scale);
        const float cS = pow2i(-ez) * pow2i(-ez) * p.scale * kL2E;  // s2 = (x.y 2^2e) cS
        const float inv = pow2i(-E) * pow2i(-ez);                  // a dZ block back to z.grad units
        const int rb_first = rb_of_tile(t_begin, p.CT);
        const int rb_last = n > 0 ? rb_of_tile(t_end - 1, p.CT) : rb_first - 1;
        float dacc[32];
#pragma unroll
        for (int f = 0; f < 32; ++f) dacc[f] = 0.f;
        float lse2k = 0.f, gk = 0.f;
        int rb_cur = rb_first, row = rb_first * kBM + lr;
        auto load_row = [&]() {
            row = rb_cur * kBM + lr;
            // rows past the stats (the last row block may pass N by more than the padding): no weight
            const float4 st = row < N32 ? p.stat[row] : make_float4(__int_as_float(0xff800000), 0.f, 0.f, 0.f);
            lse2k = st.x;
            gk = st.y;
        };
        load_row();
        bool ok = true;
        // add this warp's 32 features of the group's finished dZ block of tile j into the accumulator
        auto drain = [&](int64_t j) -> bool {
            if (!mbar_wait_warp(dz_full + grp, (uint32_t)((j >> 1) & 1), p.err, 67)) return false;
            fence_after_sync();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float v[16], w[16];
                const uint32_t a = tD(grp) + lane_off + (uint32_t)(32 * half + 16 * c);
                tmem_ld16x2(a, a + 64, v, w);
#pragma unroll
                for (int u = 0; u < 16; ++u) dacc[16 * c + u] = fmaf(v[u] + w[u], inv, dacc[16 * c + u]);
            }
            fence_before_sync();
            mbar_arrive_warp(dz_empty + grp);
            return true;
        };
        // Write this thread's partial of row block rb_cur (both groups, every row block of the range in
        // order); the CTA that completes the row block merges it into z.grad.
        auto flush = [&]() {
            const int seg = rb_cur - rb_first;
            float* o = p.part + (size_t)(blockIdx.x * p.smax + seg) * kPartRowsL * kBM;
#pragma unroll
            for (int f = 0; f < 32; ++f) o[(size_t)(grp * 64 + 32 * half + f) * kBM + lr] = dacc[f];
            __threadfence();
            mbar_arrive_warp(fl_bar);
            if (etid == 0) {
                int last = 0;
                if (mbar_wait(fl_bar, (uint32_t)(seg & 1), p.err, 68)) {
                    const int64_t t0 = (int64_t)rb_cur * p.CT;
                    const int need = cta_of_tile(p.T, p.G, t0 + p.CT - 1) - cta_of_tile(p.T, p.G, t0) + 1;
                    last = atomicAdd(p.cnt + rb_cur, 1) + 1 == need;
                    __threadfence();
                }
                *sflag = last;
                mbar_arrive(dec_bar);
            }
            if (mbar_wait_warp(dec_bar, (uint32_t)(seg & 1), p.err, 69) && *sflag)
                lin_merge_row(p, rb_cur, etid % kBM, etid / kBM);
#pragma unroll
            for (int f = 0; f < 32; ++f) dacc[f] = 0.f;
        };
        int64_t pending = -1;
        TileCursor cur(t_begin, p.CT);
        if (grp == 1 && n > 0) cur.next();
        for (int64_t i = grp; i < n && ok; i += 2, cur.next(), cur.next()) {
            const int rb = cur.rb, ct = cur.ct;
            if (rb != rb_cur) {
                if (pending >= 0) {
                    ok = drain(pending);
                    pending = -1;
                    if (!ok) break;
                }
                while (rb_cur < rb) {
                    flush();
                    ++rb_cur;
                }
                load_row();
            }
            const int s = (int)(i % kStagesS);
            ok = mbar_wait_warp(s_full + grp, (uint32_t)((i >> 1) & 1), p.err, 70) &&
                 mbar_wait_warp(bs_full + s, (uint32_t)((i / kStagesS) & 1), p.err, 71);  // the tile's column stats
            if (!ok) break;
            fence_after_sync();
            const int dead_self = p.exclude_self ? row : -1;  // the pair (row, row)
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                const int ks = 2 * half + c;
                const uint32_t col = tS(grp) + lane_off + (uint32_t)(16 * ks);
                float v[16], w[16];
                tmem_ld16x2(col, col + 64, v, w);  // hi*hi, hi*lo + lo*hi
                const float4* st = sStat + s * kBNb + 16 * ks;
                // kappa 2^E = a_k 2^(s2 + E - lse2_k) + a_j 2^(s2 + E - lse2_j), a = scale g; row and column
                // stats alike are (E - lse2, a)
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float2 cc = *reinterpret_cast<const float2*>(st + u);
                    const float t = v[u] + w[u];
                    v[u] = fmaf(gk, ExpTraits<float>::bexp(fmaf(t, cS, lse2k)), cc.y * ExpTraits<float>::bexp(fmaf(t, cS, cc.x)));
                }
                const int j0 = ct * kBNb + 16 * ks;
                const int lim = N32 - j0, self = dead_self - j0;  // columns u >= lim are padding
                if (__any_sync(0xffffffffu, lim < 16 || (self >= 0 && self < 16))) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) v[u] = (u >= lim || u == self) ? 0.f : v[u];
                }
                uint32_t hw[8], lw[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const __half2 h = __floats2half2_rn(v[2 * k], v[2 * k + 1]);
                    const float2 hf = __half22float2(h);
                    hw[k] = *reinterpret_cast<const uint32_t*>(&h);
                    lw[k] = pack_f16x2(v[2 * k] - hf.x, v[2 * k + 1] - hf.y);
                }
                // kappa of K step ks over this warp's own hi*hi columns [16 ks, 16 ks + 16), read above
                tmem_st8(col, hw);
                tmem_st8(col + 8, lw);
            }
            tmem_st_wait();
            fence_before_sync();
            mbar_arrive_warp(w_full + grp);
            if (pending >= 0) {
                ok = drain(pending);
                if (!ok) break;
            }
            pending = i;
        }
        if (ok && pending >= 0) ok = drain(pending);
        if (ok) {
            while (rb_cur <= rb_last) {
                flush();
                ++rb_cur;
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Backward pre-pass, one warp per row over the padded rows: the fp16 hi/lo split of z 2^e, |z|^2 and the
// column stats (lse_j log2 e, g_j, 2^-e_j, scale 2^-e_j), (+inf, 0, 0, 0) for padding rows.
__global__ void __launch_bounds__(256) lse_bwd_prep16(const float* __restrict__ z, const float* __restrict__ lse,
                                                      const float* __restrict__ g, float scale, int64_t N, int64_t Npad,
                                                      __half2* __restrict__ hi, __half2* __restrict__ lo,
                                                      float* __restrict__ zn, float4* __restrict__ stat,
                                                      int* __restrict__ cnt, int64_t ncnt) {
    griddep_wait();
    griddep_launch();
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (lane == 0 && r < ncnt) cnt[r] = 0;  // the main kernel's per-row-block arrival counters
    if (r >= Npad) return;
    if (r >= N) {
        if (lane == 0) stat[r] = make_float4(__int_as_float(0x7f800000), 0.f, 0.f, 0.f);
        return;
    }
    const float2 v = reinterpret_cast<const float2*>(z + r * 64)[lane];
    float m = fmaxf(fabsf(v.x), fabsf(v.y)), ss = fmaf(v.x, v.x, v.y * v.y);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    }
    const int e = f16_row_exponent(m);
    const float f = pow2i(e);
    const float a = v.x * f, b = v.y * f;
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    hi[r * 32 + lane] = h;
    lo[r * 32 + lane] = __floats2half2_rn(a - hf.x, b - hf.y);
    if (lane == 0) {
        zn[r] = ss;
        stat[r] = make_float4(lse[r] * 1.4426950408889634f, g[r], pow2i(-e), scale * pow2i(-e));
    }
}

// Linear score without exp: the largest |z| and |g| (float bits, combined with atomicMax; both are
// non-negative) for the sweep's two powers of two. One warp per row, grid-stride; one atomic per block.
__global__ void __launch_bounds__(256) lse_bwd_reduce(const float* __restrict__ z, const float* __restrict__ g,
                                                      int64_t N, int* __restrict__ gm) {
    griddep_wait();
    griddep_launch();
    __shared__ float red[2][8];
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float mz = 0.f, mg = 0.f;
    const int64_t stride = (int64_t)gridDim.x * 8;
    // eight rows' loads in flight per warp before any is used (the data comes from DRAM)
    for (int64_t r0 = (int64_t)blockIdx.x * 8 + wib; r0 < N; r0 += 8 * stride) {
        float2 v[8];
        float gg[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t r = r0 + k * stride;
            v[k] = r < N ? reinterpret_cast<const float2*>(z + r * 64)[lane] : make_float2(0.f, 0.f);
            gg[k] = r < N && lane == 0 ? g[r] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            mz = fmaxf(mz, fmaxf(fabsf(v[k].x), fabsf(v[k].y)));
            mg = fmaxf(mg, fabsf(gg[k]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mz = fmaxf(mz, __shfl_xor_sync(0xffffffffu, mz, off));
    if (lane == 0) {
        red[0][wib] = mz;
        red[1][wib] = mg;
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        float m = 0.f;
        for (int w = 0; w < 8; ++w) m = fmaxf(m, red[threadIdx.x][w]);
        atomicMax(gm + threadIdx.x, __float_as_int(m));
    }
}

// Linear score without exp: one warp per row over the padded rows, the fp16 hi/lo split of z 2^e with
// the matrix's power of two e, and the stats (E - lse_j log2 e, scale g_j) shared by rows and columns
// (E the kappa's power of two), (-inf, 0) for padding rows.
__global__ void __launch_bounds__(256) lse_bwd_prep_lin(const float* __restrict__ z, const float* __restrict__ lse,
                                                        const float* __restrict__ g, float scale, int64_t N,
                                                        int64_t Npad, const int* __restrict__ gm,
                                                        __half2* __restrict__ hi, __half2* __restrict__ lo,
                                                        float4* __restrict__ stat, int* __restrict__ cnt, int64_t ncnt) {
    griddep_wait();
    griddep_launch();
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (lane == 0 && r < ncnt) cnt[r] = 0;  // the main kernel's per-row-block arrival counters
    if (r >= Npad) return;
    if (r >= N) {
        if (lane == 0) stat[r] = make_float4(__int_as_float(0xff800000), 0.f, 0.f, 0.f);
        return;
    }
    const float f = pow2i(lin_z_exp(gm));
    const float2 v = reinterpret_cast<const float2*>(z + r * 64)[lane];
    const float a = v.x * f, b = v.y * f;
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    hi[r * 32 + lane] = h;
    lo[r * 32 + lane] = __floats2half2_rn(a - hf.x, b - hf.y);
    if (lane == 0)
        stat[r] = make_float4((float)lin_kappa_exp(gm, scale) - lse[r] * 1.4426950408889634f, scale * g[r], 0.f, 0.f);
}

// pfx[v] = tiles of the positions before v of a masked schedule, pfx[RB] = all of them: one block, each
// thread sums a run of consecutive positions, then an inclusive scan over the threads.
__global__ void __launch_bounds__(1024) sched_prefix(const Sched sc, int64_t* __restrict__ pfx) {
    griddep_wait();
    griddep_launch();
    __shared__ int64_t run[1024];
    const int t = threadIdx.x;
    const int64_t per = (sc.RB + 1023) / 1024;
    const int64_t b = t * per, e = b + per < sc.RB ? b + per : sc.RB;
    int64_t sum = 0;
    for (int64_t v = b; v < e; ++v) sum += sched_tiles(sc, sched_rb(sc, v));
    run[t] = sum;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int64_t v = t >= off ? run[t - off] : 0;
        __syncthreads();
        run[t] += v;
        __syncthreads();
    }
    int64_t acc = t > 0 ? run[t - 1] : 0;
    for (int64_t v = b; v < e; ++v) {
        pfx[v] = acc;
        acc += sched_tiles(sc, sched_rb(sc, v));
    }
    if (t == 1023) pfx[sc.RB] = run[1023];
}

void launch_sched_prefix(const Sched& sc, int64_t* pfx, cudaStream_t s) {
    HookScope h("sched_prefix", s);
    launch_pdl(sched_prefix, dim3(1), dim3(1024), 0, s, sc, pfx);
}

struct LseTcPlan {
    int64_t Xpad, Ypad;
    int CT;
    size_t off_xh, off_xl, off_yh, off_yl, off_xs, off_ys, off_xn, off_yn, off_part, off_cnt, off_pfx, off_prow,
        off_pcol, off_sym, bytes;
};

static LseTcPlan lse_tc_plan(int64_t N, int64_t M, bool same) {
    LseTcPlan pl;
    const int64_t RB = (N + kBM - 1) / kBM;
    pl.CT = (int)((M + kBN - 1) / kBN);
    pl.Xpad = RB * kBM;
    pl.Ypad = (int64_t)pl.CT * kBN;
    size_t o = 0;
    pl.off_xh = o; o += al256((size_t)N * kRowBytes);
    pl.off_xl = o; o += al256((size_t)N * kRowBytes);
    pl.off_xs = o; o += al256((size_t)(same ? (pl.Xpad > pl.Ypad ? pl.Xpad : pl.Ypad) : pl.Xpad) * 4);
    pl.off_xn = o; o += al256((size_t)(same ? (pl.Xpad > pl.Ypad ? pl.Xpad : pl.Ypad) : pl.Xpad) * 4);
    if (same) {
        pl.off_yh = pl.off_xh;
        pl.off_yl = pl.off_xl;
        pl.off_ys = pl.off_xs;
        pl.off_yn = pl.off_xn;
    } else {
        pl.off_yh = o; o += al256((size_t)M * kRowBytes);
        pl.off_yl = o; o += al256((size_t)M * kRowBytes);
        pl.off_ys = o; o += al256((size_t)pl.Ypad * 4);
        pl.off_yn = o; o += al256((size_t)pl.Ypad * 4);
    }
    pl.off_part = o; o += al256((size_t)(RB + kGrid) * 4 * 2 * kBM * 4);  // slot rb + CTA
    pl.off_cnt = o; o += al256((size_t)RB * 4);
    pl.off_pfx = o; o += al256((size_t)(RB + 1) * 8);
    // the symmetric sweep (lse_fwd_sym_tc) when the points are shared and its column partials stay small
    const bool symw = same && RB <= kSymCap;
    pl.off_prow = o; o += symw ? al256((size_t)(RB + kGrid) * kBM * 4 * 4) : 0;
    pl.off_pcol = o; o += symw ? al256((size_t)(RB * (RB + 1) / 2) * kBM * 4 * 4) : 0;
    pl.off_sym = o; o += symw ? 256 : 0;
    pl.bytes = o;
    return pl;
}

struct LseBwdTcPlan {
    int64_t T, Npad;
    int CT, G, smax;
    size_t off_zh, off_zl, off_zn, off_stat, off_part, off_cnt, off_gmax, bytes;
};

static LseBwdTcPlan lse_bwd_tc_plan(int64_t N) {
    LseBwdTcPlan pl;
    const int64_t RB = (N + kBM - 1) / kBM;
    pl.CT = (int)((N + kBNb - 1) / kBNb);
    pl.Npad = (int64_t)pl.CT * kBNb;
    pl.T = RB * pl.CT;
    pl.G = capped_grid((int)(pl.T < kGrid ? pl.T : kGrid));  // at most one CTA per SM of this device
    const int64_t per = (pl.T + pl.G - 1) / pl.G;
    pl.smax = (int)((per + pl.CT - 1) / pl.CT + 1);
    size_t o = 0;
    pl.off_zh = o; o += al256((size_t)N * kRowBytes);
    pl.off_zl = o; o += al256((size_t)N * kRowBytes);
    pl.off_zn = o; o += al256((size_t)N * 4);
    pl.off_stat = o; o += al256((size_t)pl.Npad * 16);
    pl.off_part = o; o += al256((size_t)pl.G * pl.smax * (kPartRowsB > kPartRowsL ? kPartRowsB : kPartRowsL) * kBM * 4);
    pl.off_cnt = o; o += al256((size_t)RB * 4);
    pl.off_gmax = o; o += 256;
    pl.bytes = o;
    return pl;
}

}  // namespace tc

size_t lse_tc_workspace(int64_t N, int64_t M, bool same) { return tc::lse_tc_plan(N, M, same).bytes; }

int launch_lse_tc(const SweepArgs& a, void* lse, bool same, cudaStream_t s) {
    using namespace tc;
    const LseTcPlan pl = lse_tc_plan(a.nP, a.nQ, same);
    int* err = device_error_word();
    if (!err) return -3;
    char* ws = static_cast<char*>(a.ws);
    __half2* xh = reinterpret_cast<__half2*>(ws + pl.off_xh);
    __half2* xl = reinterpret_cast<__half2*>(ws + pl.off_xl);
    __half2* yh = reinterpret_cast<__half2*>(ws + pl.off_yh);
    __half2* yl = reinterpret_cast<__half2*>(ws + pl.off_yl);
    float* xs = reinterpret_cast<float*>(ws + pl.off_xs);
    float* ys = reinterpret_cast<float*>(ws + pl.off_ys);
    float* xn = reinterpret_cast<float*>(ws + pl.off_xn);
    float* yn = reinterpret_cast<float*>(ws + pl.off_yn);
    int* cnt = reinterpret_cast<int*>(ws + pl.off_cnt);
    CUtensorMap mxh, mxl, myh, myl;
    if (!make_map_f16(&mxh, xh, a.nP, kBM) || !make_map_f16(&mxl, xl, a.nP, kBM) ||
        !make_map_f16(&myh, yh, a.nQ, kBN) || !make_map_f16(&myl, yl, a.nQ, kBN))
        return -1;
    int n = 0;
    const int64_t xrows = same ? (pl.Xpad > pl.Ypad ? pl.Xpad : pl.Ypad) : pl.Xpad;
    {
        HookScope h("tc_split16", s);
        launch_pdl(tc_split16, dim3((unsigned)((xrows + 7) / 8)), dim3(256), 0, s, static_cast<const float*>(a.P), a.nP,
                   xrows, xh, xl, xs, xn, cnt, (int64_t)(pl.Xpad / kBM));
        ++n;
    }
    if (!same) {
        HookScope h("tc_split16", s);
        launch_pdl(tc_split16, dim3((unsigned)((pl.Ypad + 7) / 8)), dim3(256), 0, s, static_cast<const float*>(a.Q),
                   a.nQ, pl.Ypad, yh, yl, ys, yn, (int*)nullptr, (int64_t)0);
        ++n;
    }
    // causal or band only (callers route same-group masks to the streamed sweeps): the row blocks stream
    // the column tiles that hold their kept pairs
    int64_t* pfx = reinterpret_cast<int64_t*>(ws + pl.off_pfx);
    const Sched sc = make_sched(a.pm, 0, a.band, a.nP, a.nQ, kBM, kBN, a.pm ? pfx : nullptr);
    if (a.pm) {
        launch_sched_prefix(sc, pfx, s);
        ++n;
    }
    // X = Y, linear score without exp, no mask, a triangle small enough: the symmetric sweep first; it
    // falls back (flag) to the full sweep below when the scores span too wide a range
    const int RB = (int)(pl.Xpad / kBM);
    const bool sym = same && a.metric == kLinear && !a.apply_exp && !a.pm && RB <= kSymCap;
    LseSymParams q;
    if (sym) {
        q.N = a.nP;
        q.RB = RB;
        q.T = (int64_t)RB * (RB + 1) / 2;
        q.G = capped_grid((int)(q.T < kGrid ? q.T : kGrid));
        q.exclude_self = a.exclude_self;
        q.scale = (float)a.scale;
        q.xs = xs;
        q.xn = xn;
        q.prow = reinterpret_cast<float*>(ws + pl.off_prow);
        q.pcol = reinterpret_cast<float*>(ws + pl.off_pcol);
        q.sym = reinterpret_cast<int*>(ws + pl.off_sym);
        q.err = err;
        cudaFuncSetAttribute(lse_fwd_sym_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemS);
        HookScope h("lse_fwd_sym_tc", s);
        launch_pdl(lse_fwd_sym_tc, dim3(q.G), dim3(kTcThreads), kSmemS, s, mxh, mxl, q);
        ++n;
    }
    const int64_t T = sched_total(sc);
    const int G = capped_grid((int)(T < kGrid ? T : kGrid));
    LseTcParams p;
    p.N = a.nP;
    p.M = a.nQ;
    p.sc = sc;
    p.T = T;
    p.G = G;
    p.metric = a.metric;
    p.apply_exp = a.apply_exp;
    p.exclude_self = a.exclude_self;
    p.same = same ? 1 : 0;
    p.scale = (float)a.scale;
    p.neg_gamma_log2 = (float)(-a.gamma * 1.4426950408889634);
    p.xs = xs;
    p.ys = ys;
    p.xn = xn;
    p.yn = yn;
    p.part = reinterpret_cast<float*>(ws + pl.off_part);
    p.cnt = cnt;
    p.lse = static_cast<float*>(lse);
    p.err = err;
    p.sym = sym ? q.sym : nullptr;
    p.prow = sym ? q.prow : nullptr;
    p.pcol = sym ? q.pcol : nullptr;
    p.Gs = sym ? q.G : 0;
    auto go = [&](auto kernel) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemF);
        HookScope h("lse_fwd_tc", s);
        launch_pdl(kernel, dim3(G), dim3(kTcThreads), kSmemF, s, mxh, mxl, myh, myl, p);
    };
    const bool ex = a.apply_exp != 0;
    if (a.metric == kLinear) ex ? go(lse_fwd_tc<kLinear, true>) : go(lse_fwd_tc<kLinear, false>);
    else if (a.metric == kSqeuclidean) ex ? go(lse_fwd_tc<kSqeuclidean, true>) : go(lse_fwd_tc<kSqeuclidean, false>);
    else ex ? go(lse_fwd_tc<kRbf, true>) : go(lse_fwd_tc<kRbf, false>);
    ++n;
    return n;
}

size_t lse_bwd_tc_workspace(int64_t N) { return tc::lse_bwd_tc_plan(N).bytes; }

int launch_lse_bwd_sym_tc(const SweepArgs& a, cudaStream_t s) {
    using namespace tc;
    const LseBwdTcPlan pl = lse_bwd_tc_plan(a.nP);
    int* err = device_error_word();
    if (!err) return -3;
    const bool glob = a.metric == kLinear && !a.apply_exp;
    char* ws = static_cast<char*>(a.ws);
    __half2* zh = reinterpret_cast<__half2*>(ws + pl.off_zh);
    __half2* zl = reinterpret_cast<__half2*>(ws + pl.off_zl);
    float* zn = reinterpret_cast<float*>(ws + pl.off_zn);
    float4* stat = reinterpret_cast<float4*>(ws + pl.off_stat);
    int* cnt = reinterpret_cast<int*>(ws + pl.off_cnt);
    CUtensorMap mah, mal, mbh, mbl;
    if (!make_map_f16(&mah, zh, a.nP, kBM) || !make_map_f16(&mal, zl, a.nP, kBM) ||
        !make_map_f16(&mbh, zh, a.nP, kBNb) || !make_map_f16(&mbl, zl, a.nP, kBNb))
        return -1;
    int n = 0;
    int* gm = reinterpret_cast<int*>(ws + pl.off_gmax);
    // linear score without exp: one power of two for z and one for kappa, fixed for the whole sweep (a
    // reduction finds max|z| and max|g|), and the two-group kernel lse_bwd_lin_tc; otherwise per-row powers
    // of two and lse_bwd_sym_tc with its per-tile row-maximum exchange
    if (glob) {
        cudaMemsetAsync(gm, 0, 2 * sizeof(int), s);
        {
            HookScope h("lse_bwd_reduce", s);
            const int64_t blocks = (a.nP + 7) / 8;  // one block per SM at most: few atomics on the two slots
            const int rg = capped_grid(kGrid);
            launch_pdl(lse_bwd_reduce, dim3((unsigned)(blocks < rg ? blocks : rg)), dim3(256), 0, s,
                       static_cast<const float*>(a.P), static_cast<const float*>(a.glse), a.nP, gm);
            ++n;
        }
        HookScope h("lse_bwd_prep_lin", s);
        launch_pdl(lse_bwd_prep_lin, dim3((unsigned)((pl.Npad + 7) / 8)), dim3(256), 0, s,
                   static_cast<const float*>(a.P), static_cast<const float*>(a.lse), static_cast<const float*>(a.glse),
                   (float)a.scale, a.nP, pl.Npad, (const int*)gm, zh, zl, stat, cnt, (int64_t)((a.nP + kBM - 1) / kBM));
        ++n;
    } else {
        HookScope h("lse_bwd_prep16", s);
        launch_pdl(lse_bwd_prep16, dim3((unsigned)((pl.Npad + 7) / 8)), dim3(256), 0, s,
                   static_cast<const float*>(a.P), static_cast<const float*>(a.lse), static_cast<const float*>(a.glse),
                   (float)a.scale, a.nP, pl.Npad, zh, zl, zn, stat, cnt, (int64_t)((a.nP + kBM - 1) / kBM));
        ++n;
    }
    LseBwdTcParams p;
    p.N = a.nP;
    p.T = pl.T;
    p.CT = pl.CT;
    p.G = pl.G;
    p.smax = pl.smax;
    p.metric = a.metric;
    p.apply_exp = a.apply_exp;
    p.exclude_self = a.exclude_self;
    p.scale = (float)a.scale;
    p.neg_gamma_log2 = (float)(-a.gamma * 1.4426950408889634);
    p.two_gamma = (float)(2.0 * a.gamma);
    p.zn = zn;
    p.stat = stat;
    p.part = reinterpret_cast<float*>(ws + pl.off_part);
    p.cnt = cnt;
    p.z = static_cast<const float*>(a.P);
    p.grad = static_cast<float*>(a.gP);
    p.gmax = gm;
    p.err = err;
    // the timer names the kernel actually launched
    auto go = [&](auto kernel) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemB);
        HookScope h(glob ? "lse_bwd_lin_tc" : "lse_bwd_sym_tc", s);
        launch_pdl(kernel, dim3(pl.G), dim3(kTcThreads), kSmemB, s, mah, mal, mbh, mbl, p);
    };
    const bool ex = a.apply_exp != 0;
    if (glob) go(lse_bwd_lin_tc);
    else if (a.metric == kLinear) go(lse_bwd_sym_tc<kLinear, true>);
    else if (a.metric == kSqeuclidean) ex ? go(lse_bwd_sym_tc<kSqeuclidean, true>) : go(lse_bwd_sym_tc<kSqeuclidean, false>);
    else ex ? go(lse_bwd_sym_tc<kRbf, true>) : go(lse_bwd_sym_tc<kRbf, false>);
    ++n;
    return n;
}

}  // namespace tp
