// Row top-k on the Blackwell tensor cores (fp32 data, D <= 64, no row/column parameters): torchpairwise
// guide "Using Torchpairwise in Models", Task Map (k-NN / retrieval row: lazy(X, R, "sqeuclidean")
// .topk(k, largest=False), fused, exact tie order; argmin and min are k = 1).
//
// The contraction X R^T runs on tcgen05.mma kind::tf32 with the hi/lo split of both operands (three
// products); points whose coordinates are exact in tf32 (integers up to 2^11, for instance) have lo = 0,
// so their dot products, norms and distances are exact and the selection is bit-identical to an exact
// evaluation. For the distance metrics, where two spare feature columns exist (D <= DP - 2), the norms
// ride in the contraction: rows [x, |x|^2, 1] against columns [-2y, 1, |y|^2] give the unclamped squared
// distance |x|^2 + |y|^2 - 2 x.y straight out of the accumulator, with no per-element norm loads. The
// 128 x 128 score tile lands in TMEM; eight selection warps, two per TMEM lane quarter, each take 64 of
// its columns into registers (which frees the accumulator for the next tile), turn each value into the
// score and keep a sorted (value, index) list per row in registers, inserting only on a strict
// improvement, so equal values
// keep ascending index order. The lists of the column parts and of every unit (column chunk) of a row
// block are merged lexicographically on (value, index) by a second kernel: the result is unique.
//
// Schedule: persistent CTAs over units of (row block, chunk of column tiles) dealt round-robin (see
// UnitCursor); warp 0 loads with TMA, warp 1 issues the MMAs, warps 2..9 select.
#include <cuda.h>
#include <cuda_runtime.h>

#include "tp_args.h"
#include "tp_device.cuh"
#include "tp_launch.h"
#include "tp_tc.cuh"
#include "tp_tc_host.h"

namespace tp {
namespace tc {

constexpr int kKBM = 128, kKBN = 128;
constexpr int kKLists = 4;   // sorted lists per row and unit in the partials (the most selection parts)
constexpr int kKGrid = 152;
constexpr int kAcc = 4;      // accumulators of 128 TMEM columns: the MMA may run three tiles ahead

// selection warps: eight, two per TMEM lane quarter, each owning 64 of a tile's 128 columns. (Sixteen
// warps of 32 columns, four per quarter, measured 21% slower on the k-NN workload: 18 warps leave a thread
// 96 registers and the lists spilled; 10 warps leave 128.)
__host__ __device__ constexpr int sel_warps(int DP, int K) { return 8; }

template <int DP, int SEL>
struct TopkTcShape {
    static constexpr int kChunks = DP / 32;                 // 128-byte K chunks per operand
    static constexpr int kOperand = kChunks * 128 * 128;    // 128 rows x DP fp32
    static constexpr int kPair = 2 * kOperand;              // hi + lo
    static constexpr int kStages = DP == 32 ? (SEL == 16 ? 3 : 4) : 2;
    static constexpr int kSel = SEL;
    static constexpr int kParts = kSel / 4;
    static constexpr int kCols = kKBN / kParts;
    static constexpr int kThreads = 32 * (2 + kSel);
    static constexpr size_t kKeyBuf = (size_t)kSel * 32 * 32 * 4;  // per selection warp: 32 columns x 32 lanes
    static constexpr size_t kSmem = (size_t)kPair * (1 + kStages) + (size_t)kStages * kKBN * 4 + kKeyBuf + 256 + 1024;
    static_assert(kCols == 64, "two 32-column blocks per selection warp");
    static_assert(kSmem <= 232448, "dynamic shared memory per CTA");
};

struct TopkTcParams {
    int64_t N, M;
    int CT, G, k;
    int H, U, chunk;   // column chunks per row block, units (row block, chunk), column tiles per chunk
    int parts;         // selection parts (sorted lists) per row and unit
    int metric, apply_exp, largest;
    int fold;          // the accumulator holds |x|^2 + |y|^2 - 2 x.y (norms folded into the operands)
    float scale, neg_gamma_log2;
    const float* xn;
    const float* yn;   // padded to CT * 128 entries
    float* pv;         // [U][kKLists][K][128] keys (parts beyond `parts` unused)
    int* pi;           // same layout, column indices
    const int* lo_any; // nonzero when some point has a nonzero tf32 low part (written by the split pre-pass)
    int* err;
};

// The smaller of three floats (one instruction on this architecture).
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// The smallest of 32 values.
__device__ __forceinline__ float min32(const float (&v)[32]) {
    float m[11];
#pragma unroll
    for (int g = 0; g < 10; ++g) m[g] = fmin3(v[3 * g], v[3 * g + 1], v[3 * g + 2]);
    m[10] = fminf(v[30], v[31]);
    const float a = fmin3(m[0], m[1], m[2]), b = fmin3(m[3], m[4], m[5]), c = fmin3(m[6], m[7], m[8]);
    return fmin3(fmin3(a, b, c), m[9], m[10]);
}

// Work units are (row block, chunk of column tiles), numbered u = rb * H + chunk and dealt round-robin:
// CTA c takes u = c, c + G, c + 2G, ... At any moment the CTAs work on one "wave" of G consecutive
// units, which stream the same one or two regions of the reference set (so a tile is read from HBM
// about once per wave), and each unit owns its partial lists, so the merge needs no map from CTAs to
// row blocks. (On the k-NN workload the time did not change with this schedule: the kernel is bound
// by its selection epilogue, not by the reference set's traffic.)
struct UnitCursor {
    int u, rb, ct, ct_end;
    bool valid;
    __device__ __forceinline__ explicit UnitCursor(const TopkTcParams& p) { set(p, blockIdx.x); }
    __device__ __forceinline__ void set(const TopkTcParams& p, int uu) {
        u = uu;
        valid = u < p.U;
        if (valid) {
            rb = u / p.H;
            ct = (u - rb * p.H) * p.chunk;
            ct_end = ct + p.chunk < p.CT ? ct + p.chunk : p.CT;
        }
    }
    // next tile; true when it starts a new unit (or none is left)
    __device__ __forceinline__ bool next(const TopkTcParams& p) {
        if (++ct < ct_end) return false;
        set(p, u + p.G);
        return true;
    }
};

// The score of one accumulator value: a dot product, or with folded norms the unclamped squared distance.
template <int METRIC, bool EXP>
__device__ __forceinline__ float topk_score(float acc, bool fold, float xn, float yn, float scale, float ngl2) {
    float base;
    if (METRIC == kLinear) {
        base = acc;
    } else {
        const float d2 = fmaxf(fold ? acc : fmaf(-2.f, acc, xn + yn), 0.f);
        base = METRIC == kRbf ? ExpTraits<float>::bexp(ngl2 * d2) : d2;
    }
    const float t = scale * base;
    return EXP ? ExpTraits<float>::bexp(t * 1.4426950408889634f) : t;
}

template <int DP, int K, int METRIC, bool EXP>
__global__ void __launch_bounds__(TopkTcShape<DP, sel_warps(DP, K)>::kThreads, 1)
    topk_tc(const __grid_constant__ CUtensorMap mXh, const __grid_constant__ CUtensorMap mXl,
            const __grid_constant__ CUtensorMap mYh, const __grid_constant__ CUtensorMap mYl, const TopkTcParams p) {
    using SH = TopkTcShape<DP, sel_warps(DP, K)>;
    constexpr int kChunk = 128 * 128;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_base1024(smem_raw);
    unsigned char* sA = sm;
    unsigned char* sB = sm + SH::kPair;
    float* sYn = reinterpret_cast<float*>(sB + (size_t)SH::kPair * SH::kStages);  // [stage][128]
    float* sKeys = sYn + SH::kStages * kKBN;                                         // [warp][32 u][32 lanes]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKeys + SH::kKeyBuf / 4);
    uint64_t* a_full = bars + 0;
    uint64_t* a_empty = bars + 1;
    uint64_t* b_full = bars + 2;               // [kStages]
    uint64_t* b_empty = bars + 2 + SH::kStages;
    uint64_t* acc_full = bars + 2 + 2 * SH::kStages;   // [kAcc]
    uint64_t* acc_empty = acc_full + kAcc;             // [kAcc]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_empty + kAcc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        prefetch_map(&mXh);
        prefetch_map(&mXl);
        prefetch_map(&mYh);
        prefetch_map(&mYl);
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int s = 0; s < SH::kStages; ++s) {
            mbar_init(b_full + s, 1);
            // freed by the MMA (operands consumed) and, where the selection reads the stage's column norms
            // (norms not folded into the contraction), by the selection warps, one arrival each
            mbar_init(b_empty + s, p.fold ? 1 : 1 + SH::kSel);
        }
        for (int b = 0; b < kAcc; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, SH::kSel);
        }
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, 128 * kAcc);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer
            // with every low part zero the MMAs read only the high parts: the low tiles are not loaded
            const bool lo = *reinterpret_cast<const volatile int*>(p.lo_any) != 0;
            const uint32_t bytes = lo ? SH::kPair : SH::kOperand;
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            int64_t i = 0;
            for (UnitCursor cur(p); cur.valid && ok; ++i, cur.next(p)) {
                const int rb = cur.rb, ct = cur.ct;
                if (rb != rb_cur) {
                    if (a_uses > 0) ok = mbar_wait(a_empty, (a_uses - 1) & 1, p.err, 81);
                    if (!ok) break;
                    mbar_expect_tx(a_full, bytes);
                    for (int c = 0; c < SH::kChunks; ++c) {
                        tma_load_2d(sA + c * kChunk, &mXh, c * 32, rb * kKBM, a_full);
                        if (lo) tma_load_2d(sA + SH::kOperand + c * kChunk, &mXl, c * 32, rb * kKBM, a_full);
                    }
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % SH::kStages), r = (int)(i / SH::kStages);
                if (r >= 1) ok = mbar_wait(b_empty + s, (r - 1) & 1, p.err, 82);
                if (!ok) break;
                unsigned char* dst = sB + (size_t)s * SH::kPair;
                mbar_expect_tx(b_full + s, bytes + (p.fold ? 0 : kKBN * 4));
                for (int c = 0; c < SH::kChunks; ++c) {
                    tma_load_2d(dst + c * kChunk, &mYh, c * 32, ct * kKBN, b_full + s);
                    if (lo) tma_load_2d(dst + SH::kOperand + c * kChunk, &mYl, c * 32, ct * kKBN, b_full + s);
                }
                if (!p.fold) bulk_load(sYn + s * kKBN, p.yn + (size_t)ct * kKBN, kKBN * 4, b_full + s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            constexpr uint32_t idesc = idesc_tf32(kKBM, kKBN);
            // every low part zero (points exact in tf32, integers for instance): the two products with a low
            // part add exact zeros, so only Xh Yh is issued (the same result, a third of the MMAs)
            const int prod0 = *reinterpret_cast<const volatile int*>(p.lo_any) ? 0 : 2;
            constexpr int KS = DP / 8;
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            int64_t i = 0;
            for (UnitCursor cur(p); cur.valid && ok; ++i, cur.next(p)) {
                const int rb = cur.rb;
                if (rb != rb_cur) {
                    if (a_uses > 0) mma_commit(a_empty);
                    ok = mbar_wait(a_full, a_uses & 1, p.err, 83);
                    if (!ok) break;
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % SH::kStages), r = (int)(i / SH::kStages), b = (int)(i % kAcc), rr = (int)(i / kAcc);
                ok = mbar_wait(b_full + s, r & 1, p.err, 84);
                if (ok && rr >= 1) ok = mbar_wait(acc_empty + b, (rr - 1) & 1, p.err, 85);
                if (!ok) break;
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * kKBN);
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB + (size_t)s * SH::kPair);
                const uint32_t ao[3] = {0u, (uint32_t)SH::kOperand, 0u};  // Xh Yl, Xl Yh, then Xh Yh
                const uint32_t bo[3] = {(uint32_t)SH::kOperand, 0u, 0u};
                uint32_t acc = 0;
#pragma unroll 1
                for (int prod = prod0; prod < 3; ++prod) {
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
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
    } else {  // ---------------- selection: one row per thread, kCols of each tile per warp
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;  // column part of this warp
        const int lr = q * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * SH::kCols);
        const float sgn = p.largest ? -1.f : 1.f;
        // sqeuclidean, k smallest, no exp, positive scale: a key is scale * max(d, 0) with d the unclamped
        // distance, nondecreasing in d, so the chunk's smallest key is that of its smallest d, found with one
        // FFMA and a third of a min per element; the keys themselves are formed only when that one could
        // enter the list (the same operations, so the selection is unchanged)
        const bool fast = METRIC == kSqeuclidean && !EXP && !p.largest && p.scale > 0.f;
        float kv[K];
        int ki[K];
        float xn = 0.f;
        bool ok = true;
        auto reset = [&]() {
#pragma unroll
            for (int t = 0; t < K; ++t) {
                kv[t] = pinf<float>();
                ki[t] = 0x7fffffff;
            }
        };
        auto flush = [&](int u) {
            const size_t base = ((size_t)u * kKLists + half) * K * kKBM;
#pragma unroll
            for (int t = 0; t < K; ++t) {
                p.pv[base + (size_t)t * kKBM + lr] = kv[t];
                p.pi[base + (size_t)t * kKBM + lr] = ki[t];
            }
        };
        bool fresh = true;
        int64_t i = 0;
        for (UnitCursor cur(p); cur.valid && ok; ++i) {
            const int rb = cur.rb, ct = cur.ct;
            if (fresh) {
                reset();
                const int64_t row = (int64_t)rb * kKBM + lr;
                xn = (METRIC != kLinear && !p.fold && row < p.N) ? p.xn[row] : 0.f;
                fresh = false;
            }
            const int b = (int)(i % kAcc), rr = (int)(i / kAcc), s = (int)(i % SH::kStages);
            ok = mbar_wait_warp(acc_full + b, rr & 1, p.err, 86);
            if (!ok) break;
            fence_after_sync();
            // both 32-column blocks of this part into registers, then the accumulator goes back to the MMA
            float v[32], vn[32];
            tmem_ld32x2(lane_base + (uint32_t)(b * kKBN), lane_base + (uint32_t)(b * kKBN + 32), v, vn);
            fence_before_sync();
            mbar_arrive_warp(acc_empty + b);
            const int j0 = ct * kKBN + half * SH::kCols;
            const int lim = (int)(p.M - j0 < SH::kCols ? p.M - j0 : SH::kCols);  // valid columns of this part
            const float* yn = sYn + s * kKBN + half * SH::kCols;
            float* wkeys = sKeys + (warp - 2) * 32 * 32;
#pragma unroll 1
            for (int c = 0; c < SH::kCols / 32; ++c) {
                if (c == 1) {
#pragma unroll
                    for (int u = 0; u < 32; ++u) v[u] = vn[u];
                }
                // the columns whose key beats this row's k-th key (the threshold only falls, so every column
                // the insertion would take is in the mask)
                const float thr = kv[K - 1];
                const int left = lim - c * 32;  // valid columns of these 32
                const uint32_t valid = left >= 32 ? 0xffffffffu : (left > 0 ? (1u << left) - 1u : 0u);
                uint32_t cand = 0;
                if (fast) {
                    if (!p.fold) {
#pragma unroll
                        for (int u4 = 0; u4 < 8; ++u4) {
                            const float4 y4 = reinterpret_cast<const float4*>(yn + c * 32)[u4];
                            v[u4 * 4 + 0] = fmaf(-2.f, v[u4 * 4 + 0], xn + y4.x);  // unclamped distances
                            v[u4 * 4 + 1] = fmaf(-2.f, v[u4 * 4 + 1], xn + y4.y);
                            v[u4 * 4 + 2] = fmaf(-2.f, v[u4 * 4 + 2], xn + y4.z);
                            v[u4 * 4 + 3] = fmaf(-2.f, v[u4 * 4 + 3], xn + y4.w);
                        }
                    }
                    const float kmin = p.scale * fmaxf(min32(v), 0.f);
                    if (!__any_sync(0xffffffffu, kmin < thr)) continue;
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const float key = p.scale * fmaxf(v[u], 0.f);
                        v[u] = key;
                        cand |= key < thr ? (1u << u) : 0u;
                    }
                } else {
#pragma unroll
                    for (int u4 = 0; u4 < 8; ++u4) {
                        // with folded norms the stage holds no norms (and may already hold a later tile)
                        const float4 y4 = p.fold ? make_float4(0.f, 0.f, 0.f, 0.f)
                                                 : reinterpret_cast<const float4*>(yn + c * 32)[u4];
                        const float yv[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const int u = u4 * 4 + w;
                            const float key =
                                sgn * topk_score<METRIC, EXP>(v[u], p.fold != 0, xn, yv[w], p.scale, p.neg_gamma_log2);
                            v[u] = key;
                            cand |= key < thr ? (1u << u) : 0u;
                        }
                    }
                }
                cand &= valid;
                // rare once the lists are full: stage the keys and insert the candidates in column order
                if (__any_sync(0xffffffffu, cand != 0u)) {
#pragma unroll
                    for (int u = 0; u < 32; ++u) wkeys[u * 32 + lane] = v[u];
                    __syncwarp();
                    while (cand) {
                        const int u = __ffs(cand) - 1;
                        cand &= cand - 1u;
                        topk_insert<float, K>(kv, ki, wkeys[u * 32 + lane], j0 + c * 32 + u);
                    }
                    __syncwarp();
                }
            }
            if (!p.fold) mbar_arrive_warp(b_empty + s);
            const int u_done = cur.u;
            if (cur.next(p)) {  // the unit is complete: its lists are final
                flush(u_done);
                fresh = true;
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 128 * kAcc);
}

// Per row: the lists of every (unit, part) of its row block, merged on (key, index).
template <int K>
__global__ void topk_tc_merge(TopkTcParams p, float* __restrict__ values, int64_t* __restrict__ indices) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.N) return;
    const int rb = (int)(i / kKBM), lr = (int)(i % kKBM);
    float kv[K];
    int ki[K];
#pragma unroll
    for (int t = 0; t < K; ++t) {
        kv[t] = pinf<float>();
        ki[t] = 0x7fffffff;
    }
    for (int u = rb * p.H; u < (rb + 1) * p.H; ++u) {
        for (int h = 0; h < p.parts; ++h) {
            const size_t base = ((size_t)u * kKLists + h) * K * kKBM;
            for (int t = 0; t < p.k; ++t)
                topk_insert_lex<float, K>(kv, ki, p.pv[base + (size_t)t * kKBM + lr], p.pi[base + (size_t)t * kKBM + lr]);
        }
    }
    const float sgn = p.largest ? -1.f : 1.f;
#pragma unroll
    for (int t = 0; t < K; ++t)
        if (t < p.k) {
            values[i * p.k + t] = sgn * kv[t];
            indices[i * p.k + t] = ki[t];
        }
}

// hi/lo split of a [n, D] fp32 array into [n, DP] (zero padded), row squared norms, and (for the
// streamed set) norms padded with zeros to `npad` rows. With the norms folded into the contraction
// (aug = 1: the rows, aug = 2: the columns) the two last feature columns carry them: a row becomes
// [x, 0.., |x|^2, 1], a column [-2y, 0.., 1, |y|^2] (both parts split like every other element).
__global__ void tc_split_pad(const float* __restrict__ x, int64_t n, int D, int DP, float* __restrict__ hi,
                             float* __restrict__ lo, float* __restrict__ norm, int64_t npad, int* __restrict__ lo_any,
                             int aug) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.y + threadIdx.y;  // one warp per row
    if (r >= npad) return;
    const float mul = aug == 2 ? -2.f : 1.f;
    const int last = aug ? DP - 2 : DP;  // feature columns written in the loop
    float s = 0.f;
    bool nz = false;
    for (int f = threadIdx.x; f < DP; f += 32) {
        const float e = (r < n && f < D) ? x[r * D + f] : 0.f;
        if (r < n && f < last) {
            const float h = tf32_hi(mul * e);
            const float l = tf32_lo(mul * e, h);
            hi[r * DP + f] = h;
            lo[r * DP + f] = l;
            nz |= l != 0.f;
        }
        s = fmaf(e, e, s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (threadIdx.x == 0) norm[r] = s;
    if (aug && r < n && threadIdx.x < 2) {
        // column DP - 2 + t: the norm on one side, 1 on the other
        const float e = (threadIdx.x == 0) == (aug == 1) ? s : 1.f;
        const float h = tf32_hi(e);
        const float l = tf32_lo(e, h);
        hi[r * DP + DP - 2 + threadIdx.x] = h;
        lo[r * DP + DP - 2 + threadIdx.x] = l;
        nz |= l != 0.f;
    }
    if (__any_sync(0xffffffffu, nz) && threadIdx.x == 0) atomicOr(lo_any, 1);
}

struct TopkTcPlan {
    int CT, G, DP, KB, H, U, chunk;
    bool foldable;  // two spare feature columns: the distance metrics fold the norms into the contraction
    size_t off_xh, off_xl, off_yh, off_yl, off_xn, off_yn, off_pv, off_pi, off_flag, bytes;
};

inline TopkTcPlan topk_tc_plan(int64_t N, int64_t M, int D, int k, bool same) {
    TopkTcPlan pl;
    pl.DP = D <= 32 ? 32 : 64;
    pl.foldable = D + 2 <= pl.DP;
    pl.KB = topk_bucket(k);
    const int64_t RB = (N + kKBM - 1) / kKBM;
    pl.CT = (int)((M + kKBN - 1) / kKBN);
    // column chunks per row block: enough units for about four per CTA (balance), none empty
    const int64_t want = (4 * kKGrid + RB - 1) / RB;
    const int h0 = (int)(want < 1 ? 1 : (want > pl.CT ? pl.CT : want));
    pl.chunk = (pl.CT + h0 - 1) / h0;
    pl.H = (pl.CT + pl.chunk - 1) / pl.chunk;
    pl.U = (int)(RB * pl.H);
    pl.G = pl.U < kKGrid ? pl.U : kKGrid;
    size_t o = 0;
    pl.off_xh = o; o += al256((size_t)N * pl.DP * 4);
    pl.off_xl = o; o += al256((size_t)N * pl.DP * 4);
    if (same && !pl.foldable) {  // with folded norms the two sides differ even for the same points
        pl.off_yh = pl.off_xh;
        pl.off_yl = pl.off_xl;
    } else {
        pl.off_yh = o; o += al256((size_t)M * pl.DP * 4);
        pl.off_yl = o; o += al256((size_t)M * pl.DP * 4);
    }
    pl.off_xn = o; o += al256((size_t)N * 4);
    pl.off_yn = o; o += al256((size_t)pl.CT * kKBN * 4);
    const size_t lists = (size_t)pl.U * kKLists * pl.KB * kKBM;
    pl.off_pv = o; o += al256(lists * 4);
    pl.off_pi = o; o += al256(lists * 4);
    pl.off_flag = o; o += 256;
    pl.bytes = o;
    return pl;
}

}  // namespace tc

size_t topk_tc_workspace(int64_t N, int64_t M, int D, int k, bool same) {
    return tc::topk_tc_plan(N, M, D, k, same).bytes;
}

// Tensor-core top-k; returns the number of kernels launched or -1 (tensor maps could not be built).
int launch_topk_tc(const SweepArgs& a, void* values, int64_t* indices, bool same, cudaStream_t s) {
    using namespace tc;
    const TopkTcPlan pl = topk_tc_plan(a.nP, a.nQ, a.D, a.k, same);
    int* err = device_error_word();
    if (!err) return -3;
    char* ws = static_cast<char*>(a.ws);
    float* xh = reinterpret_cast<float*>(ws + pl.off_xh);
    float* xl = reinterpret_cast<float*>(ws + pl.off_xl);
    float* yh = reinterpret_cast<float*>(ws + pl.off_yh);
    float* yl = reinterpret_cast<float*>(ws + pl.off_yl);
    float* xn = reinterpret_cast<float*>(ws + pl.off_xn);
    float* yn = reinterpret_cast<float*>(ws + pl.off_yn);
    CUtensorMap mxh, mxl, myh, myl;
    if (!make_map_2d(&mxh, xh, pl.DP, a.nP, 128) || !make_map_2d(&mxl, xl, pl.DP, a.nP, 128) ||
        !make_map_2d(&myh, yh, pl.DP, a.nQ, 128) || !make_map_2d(&myl, yl, pl.DP, a.nQ, 128))
        return -1;
    int n = 0;
    int* lo_any = reinterpret_cast<int*>(ws + pl.off_flag);
    cudaMemsetAsync(lo_any, 0, sizeof(int), s);
    const bool fold = pl.foldable && a.metric != kLinear;
    {
        HookScope h("tc_split_pad", s);
        tc_split_pad<<<(unsigned)((a.nP + 7) / 8), dim3(32, 8), 0, s>>>(static_cast<const float*>(a.P), a.nP, a.D,
                                                                        pl.DP, xh, xl, xn, a.nP, lo_any, fold ? 1 : 0);
        ++n;
    }
    {
        // the streamed set's norms are always needed padded (the producer copies whole tiles of them)
        HookScope h("tc_split_pad", s);
        const int64_t npad = (int64_t)pl.CT * kKBN;
        tc_split_pad<<<(unsigned)((npad + 7) / 8), dim3(32, 8), 0, s>>>(static_cast<const float*>(a.Q), a.nQ, a.D,
                                                                        pl.DP, yh, yl, yn, npad, lo_any, fold ? 2 : 0);
        ++n;
    }
    TopkTcParams p;
    p.N = a.nP;
    p.M = a.nQ;
    p.CT = pl.CT;
    p.G = capped_grid(pl.G);  // units are dealt round-robin: any grid size covers them
    p.H = pl.H;
    p.U = pl.U;
    p.chunk = pl.chunk;
    p.parts = sel_warps(pl.DP, pl.KB) / 4;
    p.k = a.k;
    p.metric = a.metric;
    p.apply_exp = a.apply_exp;
    p.largest = a.largest;
    p.fold = fold ? 1 : 0;
    p.scale = (float)a.scale;
    p.neg_gamma_log2 = (float)(-a.gamma * 1.4426950408889634);
    p.xn = xn;
    p.yn = yn;
    p.pv = reinterpret_cast<float*>(ws + pl.off_pv);
    p.pi = reinterpret_cast<int*>(ws + pl.off_pi);
    p.lo_any = lo_any;
    p.err = err;
    auto go = [&](auto kernel, size_t smem) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        HookScope h("topk_tc", s);
        kernel<<<p.G, 32 * (2 + sel_warps(pl.DP, pl.KB)), smem, s>>>(mxh, mxl, myh, myl, p);
    };
    auto with_metric = [&](auto dp, auto kk) {
        constexpr int DP = decltype(dp)::value, KB = decltype(kk)::value;
        constexpr size_t sm = TopkTcShape<DP, sel_warps(DP, KB)>::kSmem;
        const bool ex = a.apply_exp != 0;
        if (a.metric == kLinear) ex ? go(topk_tc<DP, KB, kLinear, true>, sm) : go(topk_tc<DP, KB, kLinear, false>, sm);
        else if (a.metric == kSqeuclidean)
            ex ? go(topk_tc<DP, KB, kSqeuclidean, true>, sm) : go(topk_tc<DP, KB, kSqeuclidean, false>, sm);
        else ex ? go(topk_tc<DP, KB, kRbf, true>, sm) : go(topk_tc<DP, KB, kRbf, false>, sm);
    };
    auto with_k = [&](auto dp) {
        switch (pl.KB) {
            case 1: with_metric(dp, std::integral_constant<int, 1>{}); break;
            case 4: with_metric(dp, std::integral_constant<int, 4>{}); break;
            case 8: with_metric(dp, std::integral_constant<int, 8>{}); break;
            case 16: with_metric(dp, std::integral_constant<int, 16>{}); break;
            default: with_metric(dp, std::integral_constant<int, 32>{}); break;
        }
    };
    if (pl.DP == 32) with_k(std::integral_constant<int, 32>{});
    else with_k(std::integral_constant<int, 64>{});
    ++n;
    {
        HookScope h("topk_tc_merge", s);
        const unsigned nb = (unsigned)((a.nP + 127) / 128);
        switch (pl.KB) {
            case 1: topk_tc_merge<1><<<nb, 128, 0, s>>>(p, static_cast<float*>(values), indices); break;
            case 4: topk_tc_merge<4><<<nb, 128, 0, s>>>(p, static_cast<float*>(values), indices); break;
            case 8: topk_tc_merge<8><<<nb, 128, 0, s>>>(p, static_cast<float*>(values), indices); break;
            case 16: topk_tc_merge<16><<<nb, 128, 0, s>>>(p, static_cast<float*>(values), indices); break;
            default: topk_tc_merge<32><<<nb, 128, 0, s>>>(p, static_cast<float*>(values), indices); break;
        }
        ++n;
    }
    return n;
}

}  // namespace tp
