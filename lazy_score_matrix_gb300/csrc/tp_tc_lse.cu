// Row log-sum-exp on the Blackwell tensor cores (fp32 data, D = 64 features, no row/column
// parameters): torchpairwise guide "Using Torchpairwise in Models", Task Map (InfoNCE row:
// S.logsumexp(-1, exclude_self=True) on S = lazy(z, z, "linear") / t) and Score Expressions.
//
// The contraction X Y^T (D = 64) runs on tcgen05.mma kind::tf32 with a hi/lo split of both operands
// (x ~ hi + lo, hi = x with its low 13 mantissa bits cleared, lo = x - hi rounded to the nearest tf32):
// X Y^T ~ Xh Yl^T + Xl Yh^T + Xh Yh^T, which keeps fp32-level accuracy (the dropped Xl Yl^T and the
// rounding of lo are ~2^-21 relative and unbiased). The tensor core's accumulator truncates toward
// zero after each instruction, so the two small products go first: the truncations that happen at
// the full magnitude of the dot product are then only the eight of Xh Yh^T.
// The 128 x 128 score tile lands in TMEM; four epilogue warps read it back one row per thread
// (tcgen05.ld) and run the online log-sum-exp in base 2, with the metric, scale, exp and exclude_self
// applied per element. The matrix never leaves the SM.
//
// Schedule: persistent, one CTA per SM. The (row block, column tile) pairs are numbered row-block
// major and cut into equal contiguous ranges, one per CTA; a CTA's range spans at most a few row
// blocks, and for each it writes a partial (max, sum) per row. A merge kernel combines the partials
// of each row in CTA order, so results are deterministic.
//
// Warp roles (192 threads): warp 0 lane 0 loads tiles with TMA (128-byte swizzle), warp 1 owns the
// TMEM allocation and its lane 0 issues the MMAs, warps 2..5 are the epilogue. Operand ring: the row
// block's A tile (hi, lo: 64 KB) plus two stages of B tiles (hi, lo: 64 KB each); accumulators: two
// TMEM buffers of 128 columns, so the MMAs of tile i+1 overlap the epilogue of tile i.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tp_args.h"
#include "tp_device.cuh"
#include "tp_launch.h"
#include "tp_tc.cuh"
#include "tp_tc_host.h"

namespace tp {
namespace tc {

constexpr int kBM = 128;                     // rows per tile (TMEM lanes)
constexpr int kBN = 128;                     // columns per tile
constexpr int kChunk = kBM * 128;            // one 128-row x 32-fp32 swizzled chunk: 16 KB
constexpr int kOperand = 2 * kChunk;         // 64 features: two chunks, 32 KB
constexpr int kPair = 2 * kOperand;          // hi + lo: 64 KB
constexpr int kStages = 2;
constexpr int kEpiB = 16;            // backward epilogue warps: 4 per TMEM lane quarter
constexpr int kTcThreadsB = 32 * (2 + kEpiB);
constexpr int kEpiF = 16;            // forward epilogue warps: 4 per TMEM lane quarter, 32 columns each
constexpr int kTcThreadsF = 32 * (2 + kEpiF);
constexpr int kTmemCols = 256;
constexpr int kGrid = 152;                   // persistent CTAs: one per GB300 SM
constexpr size_t kSmemBytes = (size_t)kPair * (1 + kStages) + 256 + 1024;  // + barriers, + alignment slack

struct LseTcParams {
    int64_t N, M;
    int64_t T;   // total tiles = RB * CT
    int CT;      // column tiles per row block
    int G;       // CTAs
    int smax;    // partial slots per CTA
    int metric;
    int apply_exp;
    int exclude_self;
    float scale;
    float neg_gamma_log2;  // -gamma * log2(e)
    const float* xn;       // |x_i|^2 (distance metrics)
    const float* yn;       // |y_j|^2
    float* part;           // [G][smax][4 column quarters][2][128] partial (max, sum) in base 2
    int* err;
    int same;              // X and Y are the same array: the self-distance is exactly 0
};

__host__ __device__ inline int64_t range_start(int64_t T, int G, int c) { return (T * c) / G; }
// The CTA whose range holds tile t: the largest c with floor(T c / G) <= t, i.e. T c < G (t + 1).
__host__ __device__ inline int cta_of_tile(int64_t T, int G, int64_t t) { return (int)(((int64_t)G * (t + 1) - 1) / T); }

// Score of one element in base-2 units from the dot product (metric, scale, exp), or -inf.
template <int METRIC, bool EXP>
__device__ __forceinline__ float tile_score(float dot, float xn, float yn, const LseTcParams& p) {
    constexpr float kL2E = 1.4426950408889634f;
    float base;
    if (METRIC == kLinear) {
        base = dot;
    } else {
        const float d2 = fmaxf(fmaf(-2.f, dot, xn + yn), 0.f);
        base = METRIC == kRbf ? ExpTraits<float>::bexp(p.neg_gamma_log2 * d2) : d2;
    }
    const float t = p.scale * base;
    const float S = EXP ? ExpTraits<float>::bexp(t * kL2E) : t;
    return S * kL2E;
}

template <int METRIC, bool EXP>
__global__ void __launch_bounds__(kTcThreadsF, 1)
    lse_fwd_tc(const __grid_constant__ CUtensorMap mXh, const __grid_constant__ CUtensorMap mXl,
               const __grid_constant__ CUtensorMap mYh, const __grid_constant__ CUtensorMap mYl, const LseTcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = sm;                      // [hi: 2 chunks][lo: 2 chunks]
    unsigned char* sB = sm + kPair;              // stage s at sB + s * kPair
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kPair * (1 + kStages));
    uint64_t* a_full = bars + 0;
    uint64_t* a_empty = bars + 1;
    uint64_t* b_full = bars + 2;     // [kStages]
    uint64_t* b_empty = bars + 4;    // [kStages]
    uint64_t* acc_full = bars + 6;   // [2]
    uint64_t* acc_empty = bars + 8;  // [2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 10);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t_begin = range_start(p.T, p.G, blockIdx.x), t_end = range_start(p.T, p.G, blockIdx.x + 1);

    if (threadIdx.x == 0) {
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(b_full + s, 1);
            mbar_init(b_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, 32 * kEpiF);
        }
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, kTmemCols);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer
            int64_t rb_cur = -1;
            int a_uses = 0;
            bool ok = true;
            TileCursor cur(t_begin, p.CT);
            for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next()) {
                const int64_t i = t - t_begin;
                const int rb = cur.rb, ct = cur.ct;
                if (rb != rb_cur) {
                    if (a_uses > 0) ok = mbar_wait(a_empty, (a_uses - 1) & 1, p.err, 11);
                    if (!ok) break;
                    mbar_expect_tx(a_full, kPair);
                    tma_load_2d(sA, &mXh, 0, rb * kBM, a_full);
                    tma_load_2d(sA + kChunk, &mXh, 32, rb * kBM, a_full);
                    tma_load_2d(sA + kOperand, &mXl, 0, rb * kBM, a_full);
                    tma_load_2d(sA + kOperand + kChunk, &mXl, 32, rb * kBM, a_full);
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStages), r = (int)(i / kStages);
                if (r >= 1) ok = mbar_wait(b_empty + s, (r - 1) & 1, p.err, 12);
                if (!ok) break;
                unsigned char* dst = sB + s * kPair;
                mbar_expect_tx(b_full + s, kPair);
                tma_load_2d(dst, &mYh, 0, ct * kBN, b_full + s);
                tma_load_2d(dst + kChunk, &mYh, 32, ct * kBN, b_full + s);
                tma_load_2d(dst + kOperand, &mYl, 0, ct * kBN, b_full + s);
                tma_load_2d(dst + kOperand + kChunk, &mYl, 32, ct * kBN, b_full + s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            constexpr uint32_t idesc = idesc_tf32(kBM, kBN);
            int64_t rb_cur = -1;
            int a_uses = 0;
            bool ok = true;
            TileCursor cur(t_begin, p.CT);
            for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next()) {
                const int64_t i = t - t_begin;
                const int rb = cur.rb;
                if (rb != rb_cur) {
                    if (a_uses > 0) mma_commit(a_empty);  // the previous A is free once its MMAs finish
                    ok = mbar_wait(a_full, a_uses & 1, p.err, 13);
                    if (!ok) break;
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStages), r = (int)(i / kStages), b = (int)(i & 1), rr = (int)(i >> 1);
                ok = mbar_wait(b_full + s, r & 1, p.err, 14);
                if (ok && rr >= 1) ok = mbar_wait(acc_empty + b, (rr - 1) & 1, p.err, 15);
                if (!ok) break;
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * kBN);
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB + s * kPair);
                // Xh Yh^T + Xh Yl^T + Xl Yh^T over K = 64 in steps of 8 (32 bytes)
                const uint32_t ao[3] = {0u, (uint32_t)kOperand, 0u};  // Xh Yl, Xl Yh, then Xh Yh
                const uint32_t bo[3] = {(uint32_t)kOperand, 0u, 0u};
                uint32_t acc = 0;
#pragma unroll
                for (int prod = 0; prod < 3; ++prod) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t koff = (uint32_t)((ks >> 2) * kChunk + (ks & 3) * 32);
                        mma_tf32(d, desc_kmajor_sw128(a0 + ao[prod] + koff), desc_kmajor_sw128(b0 + bo[prod] + koff),
                                 idesc, acc);
                        acc = 1;
                    }
                }
                mma_commit(b_empty + s);
                mma_commit(acc_full + b);
            }
        }
    } else {  // ---------------- epilogue: warps 2..17, one row per thread, 32 of the tile's columns
        constexpr float kL2E = 1.4426950408889634f;
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int sub = (warp - 2) >> 2;        // columns [32 sub, 32 sub + 32) of each tile
        const int lr = q * 32 + lane;           // row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(sub * 32);
        // base-2 score of a plain scaled base: s = base * (scale log2 e)
        const float c1 = p.scale * kL2E;
        int64_t rb_cur = -1;
        int seg = 0;
        float m = ninf<float>(), l = 0.f, xn = 0.f;
        bool ok = true;
        auto flush = [&]() {
            float* o = p.part + ((size_t)((blockIdx.x * p.smax + seg) * 4 + sub) * 2) * kBM;
            o[lr] = m;
            o[kBM + lr] = l;
            ++seg;
        };
        TileCursor cur(t_begin, p.CT);
        for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next()) {
            const int64_t i = t - t_begin;
            const int rb = cur.rb, ct = cur.ct;
            const int64_t row = (int64_t)rb * kBM + lr;
            if (rb != rb_cur) {
                if (rb_cur >= 0) flush();
                m = ninf<float>();
                l = 0.f;
                rb_cur = rb;
                xn = (METRIC != kLinear && row < p.N) ? p.xn[row] : 0.f;
            }
            const int b = (int)(i & 1), rr = (int)(i >> 1);
            ok = mbar_wait(acc_full + b, rr & 1, p.err, 16);
            if (!ok) break;
            fence_after_sync();
            float v[32];
            tmem_ld32(lane_base + (uint32_t)(b * kBN), v);
            fence_before_sync();
            mbar_arrive(acc_empty + b);  // the values are in registers: the MMA may reuse the buffer
            const int64_t j0 = (int64_t)ct * kBN + sub * 32;
            const bool diag = row >= j0 && row < j0 + 32;
            const bool masked = p.M - j0 < 32 || (diag && (p.exclude_self || (p.same && METRIC != kLinear)));
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                float sc;
                if (METRIC == kLinear && !EXP) {
                    sc = v[u] * c1;
                } else {
                    const int64_t j = j0 + u;
                    float dot = v[u];
                    if (METRIC != kLinear && masked && p.same && j == row) dot = xn;  // |x - x|^2 = 0 exactly
                    const float yn = (METRIC != kLinear && j < p.M) ? __ldg(p.yn + j) : 0.f;
                    sc = tile_score<METRIC, EXP>(dot, xn, yn, p);
                }
                if (masked) {
                    const int64_t j = j0 + u;
                    if (j >= p.M || (p.exclude_self && j == row)) sc = ninf<float>();
                }
                v[u] = sc;
            }
            float c4[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) c4[a] = ninf<float>();
#pragma unroll
            for (int u = 0; u < 32; ++u) c4[u & 3] = fmaxf(c4[u & 3], v[u]);
            const float cmax = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));
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
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Partials of each row, in CTA order, into lse (natural log).
__global__ void lse_tc_merge(LseTcParams p, float* __restrict__ lse) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.N) return;
    const int rb = (int)(i / kBM), lr = (int)(i % kBM);
    const int64_t t0 = (int64_t)rb * p.CT, t1 = t0 + p.CT - 1;
    // first CTA whose range holds t0, last whose range holds t1 (ranges are sorted and contiguous)
    const int c_lo = cta_of_tile(p.T, p.G, t0), c_hi = cta_of_tile(p.T, p.G, t1);
    float m = ninf<float>();
    for (int c = c_lo; c <= c_hi; ++c) {
        const int seg = rb - (int)(range_start(p.T, p.G, c) / p.CT);
        for (int h = 0; h < 4; ++h) m = fmaxf(m, p.part[((size_t)((c * p.smax + seg) * 4 + h) * 2) * kBM + lr]);
    }
    float l = 0.f;
    for (int c = c_lo; c <= c_hi; ++c) {
        const int seg = rb - (int)(range_start(p.T, p.G, c) / p.CT);
        for (int h = 0; h < 4; ++h) {
            const float* o = p.part + ((size_t)((c * p.smax + seg) * 4 + h) * 2) * kBM;
            if (o[lr] > ninf<float>()) l += o[kBM + lr] * ExpTraits<float>::bexp(o[lr] - m);
        }
    }
    lse[i] = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : ninf<float>();
}

// hi/lo split of a [n, 64] fp32 array and its row squared norms.
__global__ void tc_split64(const float* __restrict__ x, int64_t n, float* __restrict__ hi, float* __restrict__ lo,
                           float* __restrict__ norm) {
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 16) + threadIdx.x / 16;  // 16 threads per row
    const int q = threadIdx.x & 15;
    if (r >= n) return;
    const float4 v = reinterpret_cast<const float4*>(x + r * 64)[q];
    float e[4] = {v.x, v.y, v.z, v.w}, h[4], lo4[4];
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        h[u] = tf32_hi(e[u]);
        lo4[u] = tf32_lo(e[u], h[u]);
        s = fmaf(e[u], e[u], s);
    }
    reinterpret_cast<float4*>(hi + r * 64)[q] = make_float4(h[0], h[1], h[2], h[3]);
    reinterpret_cast<float4*>(lo + r * 64)[q] = make_float4(lo4[0], lo4[1], lo4[2], lo4[3]);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off, 16);
    if (q == 0) norm[r] = s;
}


// ------------------------------------------------------------------------------------------------
// Symmetric backward (X = Y = z, no row/column parameters): z.grad_k = sum_j kappa_kj z_j
// - [distance metric] z_k sum_j kappa_kj, with kappa_kj the coefficient of z_j in d/dz_k of
// g_k lse_k + g_j lse_j: G = g_k P_kj + g_j P_jk (P_kj = exp(S_kj - lse_k)), H = G (times S with
// exp), E = H * scale, kappa = E (linear), -2E (sqeuclidean), 2 gamma E base (rbf). Each pair is
// evaluated once: the replay of introduction "First derivatives replay the tiles", for both sides
// of the pair at the same time.
//
// Per 64-column tile: S = Zrows Ztile^T (tf32 hi/lo, 3 products) into TMEM; the epilogue turns S
// into kappa, splits it hi/lo and stores it back into TMEM; then dZ = kappa_hi Zh + kappa_hi Zl +
// kappa_lo Zh, with kappa as the A operand read from TMEM and the tile's feature-major copy (from a
// transposed hi/lo copy of z made by the pre-pass) as a K-major B operand. A tcgen05.mma with M = 128
// costs the same for N = 64 as for N = 128 (about 64 cycles per K step, measured on the GB300), so the
// hi and lo tiles of the B operand are stacked into one 128-row operand: each product pair that shares
// its A operand is one N = 128 MMA, with hi*hi landing in TMEM columns apart from the small products,
// which the epilogue adds in fp32. That is 32 MMAs per tile instead of 48. Each tile's dZ (128 x 64)
// lands in its own (double-buffered) TMEM block and the epilogue adds it into a per-row register
// accumulator: the tensor core's accumulation then never spans more than one tile (long accumulation
// chains in TMEM drift), and the rows' sums are two-level like everywhere else. At the end of the
// CTA's share of a row block the accumulator is written as a partial; a merge kernel adds the
// partials of each row in CTA order.
// ------------------------------------------------------------------------------------------------

constexpr int kBNb = 64;                   // columns per backward tile
constexpr int kChunkB = kBNb * 128;        // 64-row x 32-fp32 chunk: 8 KB
constexpr int kChunkPairB = 2 * kChunkB;   // [hi chunk c | lo chunk c]: one 128-row K-major operand, 16 KB
constexpr int kPairB = 2 * kChunkPairB;    // both K chunks of hi and lo: 32 KB
// Two operand rings: the point-major tile (hi, lo) feeds the S MMA and is free once S is done; the
// feature-major tile (hi, lo) and the tile's (lse, g) pairs feed dZ and the epilogue and are free once dZ
// is done, which is a whole epilogue later. Separate rings let the S operands of later tiles load
// while a tile's dZ is still waiting for its epilogue.
constexpr int kStagesS = 3;
constexpr int kStagesT = 2;
// TMEM, two buffers of each: S as [hi*hi | hi*lo + lo*hi] (128 columns), overwritten by the epilogue
// with [kappa_hi | kappa_lo]; dZ likewise as [kappa_hi*Zh | kappa_hi*Zl + kappa_lo*Zh] (128 columns).
constexpr int kTmemColsB = 512;
constexpr int kPartsB = kEpiB / 4;         // epilogue warps per lane quarter, each owning a column range
constexpr int kColsB = kBNb / kPartsB;     // tile columns (and dZ features) per epilogue warp
constexpr int kPartRowsB = 64 + kPartsB;   // rows of one partial: 64 dZ features + one kappa sum per part
static_assert(kEpiB % 4 == 0 && (kColsB == 16 || kColsB == 32), "whole lane quarters, 16 or 32 columns each");
constexpr size_t kSmemBytesB = (size_t)kPair + (size_t)kPairB * (kStagesS + kStagesT) + (size_t)kStagesT * kBNb * 8 + 256 + 1024;
static_assert(kSmemBytesB <= 232448, "dynamic shared memory per CTA");

struct LseBwdTcParams {
    int64_t N;
    int64_t T;
    int CT, G, smax;
    int metric, apply_exp, exclude_self;
    float scale, neg_gamma_log2, two_gamma;
    const float* zn;      // |z_k|^2
    const float* lse2g;   // [ceil(N/64)*64][2]: (lse_j * log2 e, g_j), padded with (+inf, 0)
    float* part;          // [G][smax][64 + kPartsB][128]: dZ features, then each part's sum of kappa, row-minor
    int* err;
};

template <int METRIC, bool EXP>
__global__ void __launch_bounds__(kTcThreadsB, 1)
    lse_bwd_sym_tc(const __grid_constant__ CUtensorMap mAh, const __grid_constant__ CUtensorMap mAl,
                   const __grid_constant__ CUtensorMap mBh, const __grid_constant__ CUtensorMap mBl,
                   const __grid_constant__ CUtensorMap mTh, const __grid_constant__ CUtensorMap mTl,
                   const LseBwdTcParams p) {
    constexpr float kL2E = 1.4426950408889634f;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = sm;                                    // row block: hi (2 chunks) | lo (2 chunks)
    unsigned char* sB = sm + kPair;                        // S ring: stage s at sB + s * kPairB, [Zh | Zl]
    unsigned char* sT = sB + (size_t)kPairB * kStagesS;    // T ring: stage s at sT + s * kPairB, [ZTh | ZTl]
    float* sStat = reinterpret_cast<float*>(sT + (size_t)kPairB * kStagesT);  // [T stage][64][2]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStat + kStagesT * kBNb * 2);
    uint64_t* a_full = bars + 0;
    uint64_t* a_empty = bars + 1;
    uint64_t* bs_full = bars + 2;                 // [kStagesS]
    uint64_t* bs_empty = bs_full + kStagesS;      // [kStagesS]
    uint64_t* bt_full = bs_empty + kStagesS;      // [kStagesT]
    uint64_t* bt_empty = bt_full + kStagesT;      // [kStagesT]
    uint64_t* s_full = bt_empty + kStagesT;       // [2]
    uint64_t* w_full = s_full + 2;                // [2]
    uint64_t* dz_full = w_full + 2;               // [2]
    uint64_t* dz_empty = dz_full + 2;             // [2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(dz_empty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t_begin = range_start(p.T, p.G, blockIdx.x), t_end = range_start(p.T, p.G, blockIdx.x + 1);

    if (threadIdx.x == 0) {
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int s = 0; s < kStagesS; ++s) {
            mbar_init(bs_full + s, 1);
            mbar_init(bs_empty + s, 1);
        }
        for (int s = 0; s < kStagesT; ++s) {
            mbar_init(bt_full + s, 1);
            mbar_init(bt_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full + b, 1);
            mbar_init(w_full + b, 32 * kEpiB);
            mbar_init(dz_full + b, 1);
            mbar_init(dz_empty + b, 32 * kEpiB);
        }
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, kTmemColsB);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem, tDZ = tmem + 256;

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer: S operands run one tile ahead of T operands
            int rb_cur = -1, a_uses = 0;
            const int64_t n = t_end - t_begin;
            TileCursor cs(t_begin, p.CT), cq(t_begin, p.CT);  // next S load, next T load (each in order)
            auto load_s = [&](int64_t i) -> bool {
                const int rb = cs.rb, ct = cs.ct;
                cs.next();
                if (rb != rb_cur) {
                    if (a_uses > 0 && !mbar_wait(a_empty, (a_uses - 1) & 1, p.err, 21)) return false;
                    mbar_expect_tx(a_full, kPair);
                    tma_load_2d(sA, &mAh, 0, rb * kBM, a_full);
                    tma_load_2d(sA + kChunk, &mAh, 32, rb * kBM, a_full);
                    tma_load_2d(sA + kOperand, &mAl, 0, rb * kBM, a_full);
                    tma_load_2d(sA + kOperand + kChunk, &mAl, 32, rb * kBM, a_full);
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStagesS), r = (int)(i / kStagesS);
                if (r >= 1 && !mbar_wait(bs_empty + s, (r - 1) & 1, p.err, 22)) return false;
                unsigned char* dst = sB + (size_t)s * kPairB;
                mbar_expect_tx(bs_full + s, kPairB);
                tma_load_2d(dst, &mBh, 0, ct * kBNb, bs_full + s);
                tma_load_2d(dst + kChunkB, &mBl, 0, ct * kBNb, bs_full + s);
                tma_load_2d(dst + kChunkPairB, &mBh, 32, ct * kBNb, bs_full + s);
                tma_load_2d(dst + kChunkPairB + kChunkB, &mBl, 32, ct * kBNb, bs_full + s);
                return true;
            };
            auto load_t = [&](int64_t i) -> bool {
                const int ct = cq.ct;
                cq.next();
                const int s = (int)(i % kStagesT), r = (int)(i / kStagesT);
                if (r >= 1 && !mbar_wait(bt_empty + s, (r - 1) & 1, p.err, 29)) return false;
                unsigned char* dT = sT + (size_t)s * kPairB;  // 64 feature rows x 32 points per chunk
                mbar_expect_tx(bt_full + s, kPairB + kBNb * 8);
                tma_load_2d(dT, &mTh, ct * kBNb, 0, bt_full + s);
                tma_load_2d(dT + kChunkB, &mTl, ct * kBNb, 0, bt_full + s);
                tma_load_2d(dT + kChunkPairB, &mTh, ct * kBNb + 32, 0, bt_full + s);
                tma_load_2d(dT + kChunkPairB + kChunkB, &mTl, ct * kBNb + 32, 0, bt_full + s);
                bulk_load(sStat + s * kBNb * 2, p.lse2g + (size_t)ct * kBNb * 2, kBNb * 8, bt_full + s);
                return true;
            };
            bool ok = true;
            int64_t ns = 0;  // S tiles loaded
            for (int64_t i = 0; i < n && ok; ++i) {
                while (ok && ns < n && ns <= i + 1) ok = load_s(ns++);
                if (ok) ok = load_t(i);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            constexpr uint32_t idS = idesc_tf32(kBM, kBNb);       // S: M 128, N 64 (K = 64 features)
            constexpr uint32_t idS2 = idesc_tf32(kBM, 2 * kBNb);  // S against [Zth; Ztl]: N 128
            constexpr uint32_t idZ = idesc_tf32(kBM, 64);          // dZ: M 128, N 64 features, K = 64 points
            constexpr uint32_t idZ2 = idesc_tf32(kBM, 128);        // dZ against [ZTh; ZTl]: N 128
            int a_uses = 0;
            bool ok = true;
            // dZ for tile i (kappa already in TMEM): issue once its epilogue is done, into the dZ buffer
            // the epilogue drained two tiles ago
            auto issue_dz = [&](int64_t i) -> bool {
                const int b = (int)(i & 1), s = (int)(i % kStagesT);
                if (!mbar_wait(w_full + b, (uint32_t)((i >> 1) & 1), p.err, 25)) return false;
                if (i >= 2 && !mbar_wait(dz_empty + b, (uint32_t)(((i >> 1) - 1) & 1), p.err, 26)) return false;
                if (!mbar_wait(bt_full + s, (uint32_t)((i / kStagesT) & 1), p.err, 30)) return false;
                fence_after_sync();
                const uint32_t bz = smem_u32(sT + (size_t)s * kPairB);  // feature-major tile
                const uint32_t kh = tS + (uint32_t)(b * 128), kl = kh + 64;  // kappa_hi, kappa_lo columns
                const uint32_t dz = tDZ + (uint32_t)(b * 128);
                // per 8 points: kappa_hi [ZTh; ZTl] (N 128: hi*hi into columns 0..63, hi*lo into 64..127),
                // then kappa_lo ZTh (N 64) into columns 64..127
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = bz + (uint32_t)((ks >> 2) * kChunkPairB + (ks & 3) * 32);
                    mma_tf32_ta(dz, kh + (uint32_t)(ks * 8), desc_kmajor_sw128(kb), idZ2, ks > 0 ? 1u : 0u);
                    mma_tf32_ta(dz + 64, kl + (uint32_t)(ks * 8), desc_kmajor_sw128(kb), idZ, 1u);
                }
                mma_commit(bt_empty + s);
                mma_commit(dz_full + b);
                return true;
            };
            int rb_cur = -1;
            TileCursor cur(t_begin, p.CT);
            for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next()) {
                const int64_t i = t - t_begin;
                const int rb = cur.rb;
                if (rb != rb_cur) {
                    if (a_uses > 0) mma_commit(a_empty);
                    ok = mbar_wait(a_full, a_uses & 1, p.err, 23);
                    if (!ok) break;
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStagesS), r = (int)(i / kStagesS), b = (int)(i & 1);
                ok = mbar_wait(bs_full + s, r & 1, p.err, 24);
                if (!ok) break;
                fence_after_sync();
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB + (size_t)s * kPairB);
                const uint32_t d = tS + (uint32_t)(b * 128);
                // per 8 features: Zh [Zth; Ztl] (N 128: hi*hi into columns 0..63, hi*lo into 64..127), then
                // Zl Zth (N 64) into columns 64..127. hi*hi accumulates alone, the small products together.
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t ka = (uint32_t)((ks >> 2) * kChunk + (ks & 3) * 32);
                    const uint32_t kb = b0 + (uint32_t)((ks >> 2) * kChunkPairB + (ks & 3) * 32);
                    mma_tf32(d, desc_kmajor_sw128(a0 + ka), desc_kmajor_sw128(kb), idS2, ks > 0 ? 1u : 0u);
                    mma_tf32(d + 64, desc_kmajor_sw128(a0 + kOperand + ka), desc_kmajor_sw128(kb), idS, 1u);
                }
                mma_commit(bs_empty + s);
                mma_commit(s_full + b);
                if (i > 0) ok = issue_dz(i - 1);
            }
            if (ok && t_end > t_begin) issue_dz(t_end - t_begin - 1);
        }
    } else {  // ---------------- epilogue: warps 2..2+kEpiB, kPartsB per TMEM lane quarter
        const int q = warp & 3;
        const int part = (warp - 2) >> 2;  // tile columns [kColsB part, kColsB (part + 1)), dZ features likewise
        const int lr = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int N32 = (int)p.N;
        int seg = 0;
        float K0 = 0.f, lse2k = 0.f, gk = 0.f, zn_k = 0.f;
        float dacc[kColsB];
#pragma unroll
        for (int f = 0; f < kColsB; ++f) dacc[f] = 0.f;
        bool ok = true;
        auto drain = [&](int64_t j) -> bool {  // add this part of tile j's dZ block into the row accumulator
            const int b = (int)(j & 1);
            if (!mbar_wait(dz_full + b, (uint32_t)((j >> 1) & 1), p.err, 27)) return false;
            fence_after_sync();
            float v[kColsB], w[kColsB];
            const uint32_t col = (uint32_t)(b * 128 + part * kColsB);
            tmem_ld<kColsB>(tDZ + lane_off + col, v);
            tmem_ld<kColsB>(tDZ + lane_off + col + 64, w);
#pragma unroll
            for (int u = 0; u < kColsB; ++u) dacc[u] += v[u] + w[u];
            fence_before_sync();
            mbar_arrive(dz_empty + b);
            return true;
        };
        auto write_partial = [&]() {
            float* o = p.part + (size_t)(blockIdx.x * p.smax + seg) * kPartRowsB * kBM;
#pragma unroll
            for (int f = 0; f < kColsB; ++f) o[(size_t)(part * kColsB + f) * kBM + lr] = dacc[f];
            o[(size_t)(64 + part) * kBM + lr] = K0;
            ++seg;
        };
        int rb_cur = -1, row = 0;
        int64_t pending = -1;
        TileCursor cur(t_begin, p.CT);
        for (int64_t t = t_begin; t < t_end && ok; ++t, cur.next()) {
            const int64_t i = t - t_begin;
            const int rb = cur.rb, ct = cur.ct;
            if (rb != rb_cur) {
                if (pending >= 0) {
                    ok = drain(pending);
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
                lse2k = live ? p.lse2g[2 * row] : __int_as_float(0x7f800000);
                gk = live ? p.lse2g[2 * row + 1] : 0.f;
                zn_k = (METRIC != kLinear && live) ? p.zn[row] : 0.f;
            }
            const int b = (int)(i & 1), s = (int)(i % kStagesT);
            ok = mbar_wait(s_full + b, (uint32_t)((i >> 1) & 1), p.err, 28) &&
                 mbar_wait(bt_full + s, (uint32_t)((i / kStagesT) & 1), p.err, 31);  // the tile's (lse, g)
            if (!ok) break;
            fence_after_sync();
            const int j0 = ct * kBNb + part * kColsB;
            const int lim = N32 - j0;                       // columns u >= lim are padding
            const int self = row - j0;                      // column u == self is the pair (row, row)
            const int dead_self = p.exclude_self ? self : -1;
            const float* st = sStat + s * kBNb * 2 + part * kColsB * 2;
            float ksum = 0.f;
            {
                float v[kColsB];
                const uint32_t col = (uint32_t)(b * 128 + part * kColsB);
                float lo[kColsB];
                tmem_ld<kColsB>(tS + lane_off + col, v);        // hi*hi
                tmem_ld<kColsB>(tS + lane_off + col + 64, lo);  // hi*lo + lo*hi
#pragma unroll
                for (int u = 0; u < kColsB; ++u) {
                    const float2 lg = reinterpret_cast<const float2*>(st)[u];
                    float dot = v[u] + lo[u];
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
                    const float G = gk * ExpTraits<float>::bexp(s2 - lse2k) + lg.y * ExpTraits<float>::bexp(s2 - lg.x);
                    const bool dead = u >= lim || u == dead_self;
                    const float H = EXP ? G * S : G;
                    const float E = H * p.scale;
                    float kap = METRIC == kLinear ? E : (METRIC == kSqeuclidean ? -2.f * E : p.two_gamma * E * base);
                    kap = dead ? 0.f : kap;
                    ksum += kap;
                    const float hi = tf32_hi(kap);
                    lo[u] = tf32_lo(kap, hi);
                    v[u] = hi;
                }
                tmem_st<kColsB>(tS + lane_off + col, v);         // kappa_hi
                tmem_st<kColsB>(tS + lane_off + col + 64, lo);   // kappa_lo
            }
            K0 += ksum;
            tmem_st_wait();
            fence_before_sync();
            mbar_arrive(w_full + b);
            if (pending >= 0) {
                ok = drain(pending);
                if (!ok) break;
            }
            pending = i;
        }
        if (ok && pending >= 0) ok = drain(pending);
        if (ok && rb_cur >= 0) write_partial();
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, kTmemColsB);
}

// z.grad rows from the partials (CTA order): dZ - [distance] z * sum kappa. One block per row block:
// the partials ([64 + kPartsB][128] floats each, feature-major) are read coalesced, summed in CTA order in
// registers, and transposed through shared memory so the gradient rows are written coalesced too.
constexpr int kMergeThreads = 256;
static_assert((64 * kBM) % kMergeThreads == 0 && (kPartsB * kBM) % kMergeThreads == 0, "merge thread mapping");
__global__ void __launch_bounds__(kMergeThreads) lse_bwd_tc_merge(LseBwdTcParams p, const float* __restrict__ z,
                                                                 float* __restrict__ grad) {
    __shared__ float sd[64][kBM + 1];
    __shared__ float sk[kPartsB * kBM];
    const int rb = blockIdx.x;
    const int64_t t0 = (int64_t)rb * p.CT, t1 = t0 + p.CT - 1;
    const int c_lo = cta_of_tile(p.T, p.G, t0), c_hi = cta_of_tile(p.T, p.G, t1);
    constexpr int kPer = 64 * kBM / kMergeThreads;  // 32 (feature, row) elements per thread
    float acc[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) acc[u] = 0.f;
    constexpr int kPerK = kPartsB * kBM / kMergeThreads;  // kappa sums (part, row) per thread
    float k0[kPerK];
#pragma unroll
    for (int u = 0; u < kPerK; ++u) k0[u] = 0.f;
    for (int c = c_lo; c <= c_hi; ++c) {
        const int seg = rb - (int)(range_start(p.T, p.G, c) / p.CT);
        const float* o = p.part + (size_t)(c * p.smax + seg) * kPartRowsB * kBM;
#pragma unroll
        for (int u = 0; u < kPer; ++u) acc[u] += o[u * kMergeThreads + threadIdx.x];
#pragma unroll
        for (int u = 0; u < kPerK; ++u) k0[u] += o[64 * kBM + u * kMergeThreads + threadIdx.x];
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int e = u * kMergeThreads + threadIdx.x;
        sd[e / kBM][e % kBM] = acc[u];
    }
#pragma unroll
    for (int u = 0; u < kPerK; ++u) sk[u * kMergeThreads + threadIdx.x] = k0[u];
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * kBM; e += kMergeThreads) {
        const int lr = e / 64, f = e % 64;
        const int64_t i = (int64_t)rb * kBM + lr;
        if (i >= p.N) break;  // rows only grow with e
        const float dz = sd[f][lr];
        float ks = 0.f;
#pragma unroll
        for (int q = 0; q < kPartsB; ++q) ks += sk[q * kBM + lr];
        grad[i * 64 + f] = p.metric == kLinear ? dz : dz - z[i * 64 + f] * ks;
    }
}

// Backward pre-pass over 32 points per block (block 256): the hi/lo split of z (point-major, for the
// row operand and the S tile), its squared norms, the feature-major hi/lo copy (the K-major B operand
// of dZ = kappa Z, zero for the padding points N <= j < Npad) and the (lse_j log2 e, g_j) pairs
// (+inf, 0 for padding).
__global__ void __launch_bounds__(256) lse_bwd_prep(const float* __restrict__ z, const float* __restrict__ lse,
                                                    const float* __restrict__ g, int64_t N, int64_t Npad,
                                                    float* __restrict__ zh, float* __restrict__ zl,
                                                    float* __restrict__ zn, float* __restrict__ thi,
                                                    float* __restrict__ tlo, float* __restrict__ stat) {
    __shared__ float sh[32][65], sl[32][65];
    const int64_t j0 = (int64_t)blockIdx.x * 32;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int q4 = u * 256 + threadIdx.x;  // float4 index within the 32 x 64 block
        const int r = q4 / 16, c = (q4 % 16) * 4;
        const int64_t j = j0 + r;
        const bool live = j < N;
        float4 v = live ? reinterpret_cast<const float4*>(z + j * 64)[q4 % 16] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float e[4] = {v.x, v.y, v.z, v.w};
        float h[4], l[4], ss = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            h[w] = tf32_hi(e[w]);
            l[w] = tf32_lo(e[w], h[w]);
            ss = fmaf(e[w], e[w], ss);
            sh[r][c + w] = h[w];
            sl[r][c + w] = l[w];
        }
        if (live) {
            reinterpret_cast<float4*>(zh + j * 64)[q4 % 16] = make_float4(h[0], h[1], h[2], h[3]);
            reinterpret_cast<float4*>(zl + j * 64)[q4 % 16] = make_float4(l[0], l[1], l[2], l[3]);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off, 16);
        if ((q4 % 16) == 0 && live) zn[j] = ss;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * 32; e += 256) {
        const int f = e / 32, r = e % 32;
        const int64_t j = j0 + r;
        if (j < Npad) {
            thi[(int64_t)f * Npad + j] = sh[r][f];
            tlo[(int64_t)f * Npad + j] = sl[r][f];
        }
    }
    if (threadIdx.x < 32) {
        const int64_t j = j0 + threadIdx.x;
        if (j < Npad) {
            const bool live = j < N;
            stat[2 * j] = live ? lse[j] * 1.4426950408889634f : __int_as_float(0x7f800000);
            stat[2 * j + 1] = live ? g[j] : 0.f;
        }
    }
}


struct LseTcPlan {
    int64_t T;
    int CT, G, smax;
    size_t off_xh, off_xl, off_yh, off_yl, off_xn, off_yn, off_part, off_err, bytes;
};


static LseTcPlan lse_tc_plan(int64_t N, int64_t M, bool same) {
    LseTcPlan pl;
    const int64_t RB = (N + kBM - 1) / kBM;
    pl.CT = (int)((M + kBN - 1) / kBN);
    pl.T = RB * pl.CT;
    pl.G = (int)(pl.T < kGrid ? pl.T : kGrid);
    const int64_t per = (pl.T + pl.G - 1) / pl.G;
    pl.smax = (int)((per + pl.CT - 1) / pl.CT + 1);
    size_t o = 0;
    pl.off_xh = o; o += al256((size_t)N * 64 * 4);
    pl.off_xl = o; o += al256((size_t)N * 64 * 4);
    if (same) {
        pl.off_yh = pl.off_xh;
        pl.off_yl = pl.off_xl;
    } else {
        pl.off_yh = o; o += al256((size_t)M * 64 * 4);
        pl.off_yl = o; o += al256((size_t)M * 64 * 4);
    }
    pl.off_xn = o; o += al256((size_t)N * 4);
    if (same) pl.off_yn = pl.off_xn;
    else { pl.off_yn = o; o += al256((size_t)M * 4); }
    pl.off_part = o; o += al256((size_t)pl.G * pl.smax * 4 * 2 * kBM * 4);
    pl.off_err = o; o += 256;
    pl.bytes = o;
    return pl;
}


struct LseBwdTcPlan {
    int64_t T, Npad;
    int CT, G, smax;
    size_t off_zh, off_zl, off_zth, off_ztl, off_zn, off_stat, off_part, off_err, bytes;
};

static LseBwdTcPlan lse_bwd_tc_plan(int64_t N) {
    LseBwdTcPlan pl;
    const int64_t RB = (N + kBM - 1) / kBM;
    pl.CT = (int)((N + kBNb - 1) / kBNb);
    pl.Npad = (int64_t)pl.CT * kBNb;
    pl.T = RB * pl.CT;
    pl.G = (int)(pl.T < kGrid ? pl.T : kGrid);
    const int64_t per = (pl.T + pl.G - 1) / pl.G;
    pl.smax = (int)((per + pl.CT - 1) / pl.CT + 1);
    size_t o = 0;
    pl.off_zh = o; o += al256((size_t)N * 64 * 4);
    pl.off_zl = o; o += al256((size_t)N * 64 * 4);
    pl.off_zth = o; o += al256((size_t)pl.Npad * 64 * 4);
    pl.off_ztl = o; o += al256((size_t)pl.Npad * 64 * 4);
    pl.off_zn = o; o += al256((size_t)N * 4);
    pl.off_stat = o; o += al256((size_t)pl.Npad * 8);
    pl.off_part = o; o += al256((size_t)pl.G * pl.smax * kPartRowsB * kBM * 4);
    pl.off_err = o; o += 256;
    pl.bytes = o;
    return pl;
}

}  // namespace tc

size_t lse_tc_workspace(int64_t N, int64_t M, bool same) { return tc::lse_tc_plan(N, M, same).bytes; }

// Launches the tensor-core log-sum-exp; returns the number of kernels launched, or -1 when the
// tensor maps cannot be built (the caller then reports TP_ERR_CUDA).
int launch_lse_tc(const SweepArgs& a, void* lse, bool same, cudaStream_t s) {
    using namespace tc;
    const LseTcPlan pl = lse_tc_plan(a.nP, a.nQ, same);
    char* ws = static_cast<char*>(a.ws);
    float* xh = reinterpret_cast<float*>(ws + pl.off_xh);
    float* xl = reinterpret_cast<float*>(ws + pl.off_xl);
    float* yh = reinterpret_cast<float*>(ws + pl.off_yh);
    float* yl = reinterpret_cast<float*>(ws + pl.off_yl);
    float* xn = reinterpret_cast<float*>(ws + pl.off_xn);
    float* yn = reinterpret_cast<float*>(ws + pl.off_yn);
    CUtensorMap mxh, mxl, myh, myl;
    if (!make_map(&mxh, xh, a.nP) || !make_map(&mxl, xl, a.nP) || !make_map(&myh, yh, a.nQ) ||
        !make_map(&myl, yl, a.nQ))
        return -1;
    int n = 0;
    {
        HookScope h("tc_split64", s);
        tc_split64<<<(unsigned)((a.nP + 15) / 16), 256, 0, s>>>(static_cast<const float*>(a.P), a.nP, xh, xl, xn);
        ++n;
    }
    if (!same) {
        HookScope h("tc_split64", s);
        tc_split64<<<(unsigned)((a.nQ + 15) / 16), 256, 0, s>>>(static_cast<const float*>(a.Q), a.nQ, yh, yl, yn);
        ++n;
    }
    LseTcParams p;
    p.N = a.nP;
    p.M = a.nQ;
    p.T = pl.T;
    p.CT = pl.CT;
    p.G = pl.G;
    p.smax = pl.smax;
    p.metric = a.metric;
    p.apply_exp = a.apply_exp;
    p.exclude_self = a.exclude_self;
    p.scale = (float)a.scale;
    p.neg_gamma_log2 = (float)(-a.gamma * 1.4426950408889634);
    p.xn = xn;
    p.yn = yn;
    p.part = reinterpret_cast<float*>(ws + pl.off_part);
    p.err = reinterpret_cast<int*>(ws + pl.off_err);
    p.same = same ? 1 : 0;
    auto go = [&](auto kernel) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        HookScope h("lse_fwd_tc", s);
        kernel<<<pl.G, kTcThreadsF, kSmemBytes, s>>>(mxh, mxl, myh, myl, p);
    };
    const bool ex = a.apply_exp != 0;
    if (a.metric == kLinear) ex ? go(lse_fwd_tc<kLinear, true>) : go(lse_fwd_tc<kLinear, false>);
    else if (a.metric == kSqeuclidean) ex ? go(lse_fwd_tc<kSqeuclidean, true>) : go(lse_fwd_tc<kSqeuclidean, false>);
    else ex ? go(lse_fwd_tc<kRbf, true>) : go(lse_fwd_tc<kRbf, false>);
    ++n;
    {
        HookScope h("lse_tc_merge", s);
        lse_tc_merge<<<(unsigned)((a.nP + 127) / 128), 128, 0, s>>>(p, static_cast<float*>(lse));
        ++n;
    }
    return n;
}

size_t lse_bwd_tc_workspace(int64_t N) { return tc::lse_bwd_tc_plan(N).bytes; }

// Tensor-core symmetric backward: writes the summed gradient (dX + dY) of the same points into a.gP.
// `a` is the row-side sweep arguments (P = Q = z, lse, glse, metric, scale, exp, exclude_self).
int launch_lse_bwd_sym_tc(const SweepArgs& a, cudaStream_t s) {
    using namespace tc;
    const LseBwdTcPlan pl = lse_bwd_tc_plan(a.nP);
    char* ws = static_cast<char*>(a.ws);
    float* zh = reinterpret_cast<float*>(ws + pl.off_zh);
    float* zl = reinterpret_cast<float*>(ws + pl.off_zl);
    float* zth = reinterpret_cast<float*>(ws + pl.off_zth);
    float* ztl = reinterpret_cast<float*>(ws + pl.off_ztl);
    float* zn = reinterpret_cast<float*>(ws + pl.off_zn);
    float* stat = reinterpret_cast<float*>(ws + pl.off_stat);
    CUtensorMap mah, mal, mbh, mbl, mth, mtl;
    if (!make_map(&mah, zh, a.nP) || !make_map(&mal, zl, a.nP) || !make_map_rows(&mbh, zh, a.nP, kBNb) ||
        !make_map_rows(&mbl, zl, a.nP, kBNb) || !make_map_t(&mth, zth, pl.Npad) || !make_map_t(&mtl, ztl, pl.Npad))
        return -1;
    int n = 0;
    {
        HookScope h("lse_bwd_prep", s);
        lse_bwd_prep<<<(unsigned)(pl.Npad / 32), 256, 0, s>>>(
            static_cast<const float*>(a.P), static_cast<const float*>(a.lse), static_cast<const float*>(a.glse), a.nP,
            pl.Npad, zh, zl, zn, zth, ztl, stat);
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
    p.lse2g = stat;
    p.part = reinterpret_cast<float*>(ws + pl.off_part);
    p.err = reinterpret_cast<int*>(ws + pl.off_err);
    auto go = [&](auto kernel) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesB);
        HookScope h("lse_bwd_sym_tc", s);
        kernel<<<pl.G, kTcThreadsB, kSmemBytesB, s>>>(mah, mal, mbh, mbl, mth, mtl, p);
    };
    const bool ex = a.apply_exp != 0;
    if (a.metric == kLinear) ex ? go(lse_bwd_sym_tc<kLinear, true>) : go(lse_bwd_sym_tc<kLinear, false>);
    else if (a.metric == kSqeuclidean) ex ? go(lse_bwd_sym_tc<kSqeuclidean, true>) : go(lse_bwd_sym_tc<kSqeuclidean, false>);
    else ex ? go(lse_bwd_sym_tc<kRbf, true>) : go(lse_bwd_sym_tc<kRbf, false>);
    ++n;
    {
        HookScope h("lse_bwd_tc_merge", s);
        lse_bwd_tc_merge<<<(unsigned)((a.nP + kBM - 1) / kBM), kMergeThreads, 0, s>>>(
            p, static_cast<const float*>(a.P), static_cast<float*>(a.gP));
        ++n;
    }
    return n;
}

}  // namespace tp
