// Pairwise attention out = softmax(scale Q K^T) V and its replay backward on the Blackwell tensor
// cores (fp32 data, D = C = 64, linear score without exp or row/column parameters): torchpairwise
// guide "Using Torchpairwise in Models", Task Map (attention: softmax_matmul(V) on lazy(Q, K, "linear")
// times a scale), and the introduction (first derivatives by re-evaluating the tiles).
//
// Operands. Each of Q, K, V and dO is multiplied by one power of two of its own (its largest |element|
// brought into [2^14, 2^15)) and split into hi = fp16(x 2^e) and lo = fp16(x 2^e - hi), both rounded to
// nearest: 22 significant bits for every element within 2^17 of the matrix's largest, the same as a
// per-row power of two gives within a row, and the unscale factors of S and dP become constants. A dot
// product is (xh.yh + (xh.yl + xl.yh)) 2^-(e_x + e_y), with hi*hi in TMEM columns of its own.
//
// Forward: one sweep with an online softmax. The four warps that share a row agree on its running
// maximum m (base 2) through shared memory each tile and raise it only when a tile's maximum exceeds it by
// more than 2^8 (otherwise the stale m stands), so that kappa = 2^(s2 - m + 6) <= 2^14 stays in fp16's
// range; the row's output and sum are rescaled by 2^(m_old - m_new) on the rare raise. The log-sum-exp
// comes out of the same sweep. Backward, with dO = d loss / d out, delta_i = dO_i . out_i, dP_ij = dO_i . V_j and
// dS_ij = P_ij (dP_ij - delta_i):
//   row sweep     dQ_i = scale sum_j dS_ij K_j
//   column sweep  dK_j = scale sum_i dS_ij Q_i,   dV_j = sum_i P_ij dO_i
// All three sweeps are one kernel template. A 128 x 64 tile's S (and dP) go into TMEM; the epilogue
// reads them into registers (after which the MMA refills the buffer with a later tile) and turns them
// into coefficient rows kappa, one per output, each row scaled by a power of two fixed in advance from a
// bound (P <= 1 and |dP_ij - delta_i| <= |dO_i| |V_j| + |delta_i|): P 2^14 for the P V products, and
// dS 2^E with E from the bound for the dS products, the power of two folded into the exp. kappa is
// split into fp16 hi/lo and stored into TMEM as the A operand of the output MMA, whose B operand is the
// tile's own streamed points read MN-major: no transposed copy of any matrix exists (the column sweep
// streams Q and dO and holds K and V as its row block). Each tile's output block is added into per-row
// registers (two-level accumulation); a CTA writes one partial per row block it touched, and the last
// CTA to finish a row block adds the partials in CTA order (deterministic, no atomics on the data).
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
namespace attn {

constexpr int kBM = 128;                      // rows per tile (TMEM lanes)
constexpr int kBN = 64;                       // streamed points per tile
constexpr int kRowB = 128;                    // one point: 64 fp16 features
constexpr int kHalf = kBM * kRowB;            // 128 rows of hi (or lo): 16 KB
constexpr int kTile = kBN * kRowB;            // 64 rows of hi (or lo): 8 KB
constexpr int kStage = 4 * kTile;             // [B1 hi | B1 lo | B2 hi | B2 lo]: 32 KB
constexpr int kStages = 4;
constexpr int kABytes = 4 * kHalf;            // [A1 hi | A1 lo | A2 hi | A2 lo]: 64 KB
constexpr int kEpi = 16;                      // epilogue warps: 4 per TMEM lane quarter
constexpr int kParts = kEpi / 4;              // warps per lane quarter, each owning 16 tile columns
constexpr int kCols = kBN / kParts;           // 16: one K step of the output MMA
constexpr int kThreads = 32 * (2 + kEpi);
constexpr int kGrid = 152;                    // persistent CTAs: one per GB300 SM
constexpr size_t kXm = 2 * 4 * kBM * 4;       // forward: the four parts' tile maxima per row, two tile parities
constexpr size_t kSmem = (size_t)kABytes + (size_t)kStage * kStages + (size_t)kStages * kBN * 16 + kXm + 512 + 1024;
constexpr float kKapShift = 6.f;              // forward kappa = 2^(s2 - m + 6): at most 2^14 with the lazy maximum
constexpr float kLazy = 8.f;                  // the running maximum is raised when a tile's exceeds it by more
static_assert(kSmem <= 232448, "dynamic shared memory per CTA");
static_assert(kCols == 16, "one output K step per epilogue warp");
constexpr float kL2E = 1.4426950408889634f;

// Slots of the global maxima (float bits of non-negative values, combined with atomicMax on int):
// |Q|, |K|, |V|, |dO| elementwise, the largest row norms of V and dO, the largest |delta_i|.
enum Slot : int { gQ = 0, gK, gV, gD, gVn, gDn, gDelta, kSlots };

enum Mode : int { kFwd = 0, kRowSweep = 1, kColSweep = 2 };

// Per mode: the row block holds A1 (for S) and, for the backward, A2 (for dP); a stage holds B1 (the
// other side of S) and B2 (the other side of dP, or V in the forward).
//   kFwd:      rows Q, A1 = Q;          stream B1 = K, B2 = V;   out0 = O  <- kappa0 B2
//   kRowSweep: rows Q, A1 = Q, A2 = dO; stream B1 = K, B2 = V;   out0 = dQ <- kappa0 B1
//   kColSweep: rows K, A1 = K, A2 = V;  stream B1 = Q, B2 = dO;  out0 = dK <- kappa0 B1, out1 = dV <- kappa1 B2
template <int MODE>
struct Shape {
    static constexpr bool kDP = MODE != kFwd;                       // dP = A2 B2^T is formed
    static constexpr int kOuts = MODE == kColSweep ? 2 : 1;
    static constexpr int kRegion = kDP ? 256 : 128;                 // TMEM columns of one S (+ dP) buffer
    static constexpr int kBuf = kDP ? 1 : 2;                        // S (+ dP) buffers
    static constexpr bool kColStats = MODE == kColSweep;            // the stage carries per-column stats
    static constexpr int kF = 64 * kOuts;                           // features of one partial row
    // rows of one partial: the features, and for the forward the row maximum and the four parts' sums
    static constexpr int kPartRows = MODE == kFwd ? kF + 1 + kParts : kF;
    // One output: kappa_hi [B_hi | B_lo] (N 128, hi*hi and hi*lo in 128 accumulator columns) and
    // kappa_lo B_hi (N 64) into the hi*lo half. Two outputs (column sweep): TMEM holds one 64-column
    // accumulator each, fed by three N 64 MMAs.
    static constexpr bool kWide = kOuts == 1;
    static constexpr int kAccW = kWide ? 128 : 64;
    // TMEM column of output o's kappa (hi in +0..31, lo in +32..63) and accumulator
    __host__ __device__ static constexpr uint32_t kap(int o) { return (uint32_t)(kBuf * kRegion + 64 * o); }
    __host__ __device__ static constexpr uint32_t acc(int o) { return (uint32_t)(kBuf * kRegion + 64 * kOuts + kAccW * o); }
    // the stage part that is the B operand of output o
    __host__ __device__ static constexpr uint32_t out_b(int o) {
        return MODE == kRowSweep ? 0u : (o == 0 && MODE == kColSweep ? 0u : 2u * kTile);
    }
};
static_assert(Shape<kColSweep>::acc(1) + 64 <= 512 && Shape<kRowSweep>::acc(0) + 128 <= 512 &&
                  Shape<kFwd>::acc(0) + 128 <= 512,
              "TMEM columns");

struct Params {
    int64_t R;             // rows of the sweep (queries; keys for the column sweep)
    int64_t C;             // streamed points (keys; queries for the column sweep)
    Sched sc;              // the tiles each row block streams (all CT of them without a pair mask)
    int64_t T;             // tiles
    int G;
    float scale;
    const float4* rstat;   // [rows padded to 128] the row side's stats
    const float4* cstat;   // [CT * 64 or more] the streamed side's stats (column sweep)
    const int* gmax;       // [kSlots] the global maxima
    float* part;           // [RB + G][F][128] partials, slot position + CTA, row-minor
    int* cnt;              // [row blocks] CTAs done with each row block (zeroed by the pre-pass)
    float* out0;           // [R][64] (null: not wanted)
    float* out1;
    int acc0;              // add output 0 into out0 instead of writing it
    float* lse;            // forward: the row log-sum-exp [R]
    int* err;
};

// The power of two of a matrix from its largest |element| (the same rule as per row elsewhere).
__device__ __forceinline__ int gexp(const int* gm, int slot) { return f16_row_exponent(__int_as_float(__ldg(gm + slot))); }

// Output features [FG fg, FG fg + FG) of row lr of row block rb: the partials of every CTA that saw the
// row block, added in CTA order.
template <int MODE>
__device__ __noinline__ void merge_row(const Params& p, int rb, int lr, int fg) {
    using SH = Shape<MODE>;
    constexpr int FG = SH::kF / 4;
    const int64_t row = (int64_t)rb * kBM + lr;
    if (row >= p.R) return;
    const int fb = fg * FG;
    float* dst = fb < 64 ? p.out0 : p.out1;
    if (!dst) return;
    const int64_t v = sched_pos(p.sc, rb), t0 = tile_start(p.sc, v), t1 = tile_start(p.sc, v + 1) - 1;
    const int c_lo = cta_of_tile(p.T, p.G, t0), c_hi = cta_of_tile(p.T, p.G, t1);
    float acc[FG];
#pragma unroll
    for (int f = 0; f < FG; ++f) acc[f] = 0.f;
    float4* d4 = reinterpret_cast<float4*>(dst + row * 64 + (fb & 63));
    if constexpr (MODE == kFwd) {
        // each CTA's part in its own frame: maximum m_c, sum l_c (four parts), output sums; in CTA order
        float M = ninf<float>();
        for (int c = c_lo; c <= c_hi; ++c) M = fmaxf(M, __ldcg(p.part + ((size_t)(v + c) * SH::kPartRows + SH::kF) * kBM + lr));
        float L = 0.f;
        if (M != ninf<float>()) {
            for (int c = c_lo; c <= c_hi; ++c) {
                const float* o = p.part + (size_t)(v + c) * SH::kPartRows * kBM + lr;
                const float mc = __ldcg(o + (size_t)SH::kF * kBM);
                if (mc == ninf<float>()) continue;
                const float w = ExpTraits<float>::bexp(mc - M);
                float lc = 0.f;
#pragma unroll
                for (int h = 0; h < kParts; ++h) lc += __ldcg(o + (size_t)(SH::kF + 1 + h) * kBM);
                L = fmaf(w, lc, L);
#pragma unroll
                for (int f = 0; f < FG; ++f) acc[f] = fmaf(w, __ldcg(o + (size_t)(fb + f) * kBM), acc[f]);
            }
        }
        const float invL = L > 0.f ? 1.f / L : 0.f;  // a row with every pair masked returns 0
#pragma unroll
        for (int f4 = 0; f4 < FG / 4; ++f4)
            d4[f4] = make_float4(acc[4 * f4] * invL, acc[4 * f4 + 1] * invL, acc[4 * f4 + 2] * invL, acc[4 * f4 + 3] * invL);
        // kappa carries 2^(6 - m): sum_j 2^(s2_j) = L 2^(M - 6)
        if (fg == 0 && p.lse) p.lse[row] = L > 0.f ? ExpTraits<float>::lse(M - kKapShift, L) : ninf<float>();
        return;
    }
    for (int c = c_lo; c <= c_hi; ++c) {
        const float* o = p.part + (size_t)(v + c) * SH::kPartRows * kBM + lr;
#pragma unroll
        for (int f = 0; f < FG; ++f) acc[f] += __ldcg(o + (size_t)(fb + f) * kBM);
    }
    const bool add = p.acc0 && fb < 64;
#pragma unroll
    for (int f4 = 0; f4 < FG / 4; ++f4) {
        float4 v = make_float4(acc[4 * f4], acc[4 * f4 + 1], acc[4 * f4 + 2], acc[4 * f4 + 3]);
        if (add) {
            const float4 o = d4[f4];
            v = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
        }
        d4[f4] = v;
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc(const __grid_constant__ CUtensorMap mA1h, const __grid_constant__ CUtensorMap mA1l,
            const __grid_constant__ CUtensorMap mA2h, const __grid_constant__ CUtensorMap mA2l,
            const __grid_constant__ CUtensorMap mB1h, const __grid_constant__ CUtensorMap mB1l,
            const __grid_constant__ CUtensorMap mB2h, const __grid_constant__ CUtensorMap mB2l, const Params p) {
    using SH = Shape<MODE>;
    constexpr int NB = SH::kBuf;
    constexpr int NO = SH::kOuts;
    constexpr bool CST = SH::kColStats;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_base1024(smem_raw);
    unsigned char* sA = sm;
    unsigned char* sB = sm + kABytes;
    float4* sStat = reinterpret_cast<float4*>(sB + (size_t)kStage * kStages);   // [stage][64]
    float* xm = reinterpret_cast<float*>(sStat + kStages * kBN);                // forward: [2][4 parts][128 rows]
    uint64_t* bars = reinterpret_cast<uint64_t*>(xm + kXm / 4);
    uint64_t* a_full = bars + 0;
    uint64_t* a_empty = bars + 1;
    uint64_t* bs_full = bars + 2;              // [kStages]
    uint64_t* bs_empty = bs_full + kStages;    // [kStages]
    uint64_t* s_full = bs_empty + kStages;     // [NB] S (and dP) of a buffer are in TMEM
    uint64_t* s_free = s_full + NB;            // [NB] the epilogue has read the buffer into registers
    uint64_t* w_full = s_free + NB;            // the epilogue stored the tile's kappa
    uint64_t* o_full = w_full + 1;             // the output MMAs of a tile finished
    uint64_t* fl_bar = o_full + 1;             // the epilogue wrote its partials of a row block
    uint64_t* dec_bar = fl_bar + 1;            // the CTA knows whether it merges that row block
    uint64_t* x_bar = dec_bar + 1;             // forward: [4 quarters][2 parities] the quarter's tile maxima are in xm
    uint32_t* tslot = reinterpret_cast<uint32_t*>(x_bar + 8);
    volatile int* sflag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t_begin = range_start(p.T, p.G, blockIdx.x), t_end = range_start(p.T, p.G, blockIdx.x + 1);
    const int64_t n = t_end - t_begin;

    if (threadIdx.x == 0) {
        prefetch_map(&mA1h);
        prefetch_map(&mA1l);
        prefetch_map(&mA2h);
        prefetch_map(&mA2l);
        prefetch_map(&mB1h);
        prefetch_map(&mB1l);
        prefetch_map(&mB2h);
        prefetch_map(&mB2l);
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bs_full + s, 1);
            mbar_init(bs_empty + s, 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(s_full + b, 1);
            mbar_init(s_free + b, 32 * kEpi);
        }
        mbar_init(w_full, 32 * kEpi);
        mbar_init(o_full, 1);
        mbar_init(fl_bar, 32 * kEpi);
        mbar_init(dec_bar, 1);
        for (int x = 0; x < 8; ++x) mbar_init(x_bar + x, kParts);  // one arrival per warp of the quarter
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    griddep_wait();

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer: row blocks and operand stages in tile order
            int rb_cur = -1, a_uses = 0;
            bool ok = true;
            SchedCursor cur(p.sc, t_begin);
            for (int64_t i = 0; i < n && ok; ++i, cur.next(p.sc)) {
                const int rb = cur.rb, ct = cur.ct;
                if (rb != rb_cur) {
                    if (a_uses > 0) ok = mbar_wait(a_empty, (a_uses - 1) & 1, p.err, 41);
                    if (!ok) break;
                    mbar_expect_tx(a_full, SH::kDP ? 4 * kHalf : 2 * kHalf);
                    tma_load_2d(sA, &mA1h, 0, rb * kBM, a_full);
                    tma_load_2d(sA + kHalf, &mA1l, 0, rb * kBM, a_full);
                    if (SH::kDP) {
                        tma_load_2d(sA + 2 * kHalf, &mA2h, 0, rb * kBM, a_full);
                        tma_load_2d(sA + 3 * kHalf, &mA2l, 0, rb * kBM, a_full);
                    }
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(i % kStages), r = (int)(i / kStages);
                if (r >= 1) ok = mbar_wait(bs_empty + s, (r - 1) & 1, p.err, 42);
                if (!ok) break;
                unsigned char* dst = sB + (size_t)s * kStage;
                mbar_expect_tx(bs_full + s, kStage + (CST ? kBN * 16 : 0));
                tma_load_2d(dst, &mB1h, 0, ct * kBN, bs_full + s);
                tma_load_2d(dst + kTile, &mB1l, 0, ct * kBN, bs_full + s);
                tma_load_2d(dst + 2 * kTile, &mB2h, 0, ct * kBN, bs_full + s);
                tma_load_2d(dst + 3 * kTile, &mB2l, 0, ct * kBN, bs_full + s);
                if (CST) bulk_load(sStat + s * kBN, p.cstat + (size_t)ct * kBN, kBN * 16, bs_full + s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            constexpr uint32_t idS2 = idesc_f16(kBM, 2 * kBN, false);  // A_hi [B_hi; B_lo]: N 128
            constexpr uint32_t idS = idesc_f16(kBM, kBN, false);       // A_lo B_hi: N 64
            constexpr uint32_t idO = idesc_f16(kBM, 64, true);         // kappa B (MN-major): N 64
            constexpr uint32_t idO2 = idesc_f16(kBM, 128, true);       // kappa_hi [B_hi | B_lo] (MN-major): N 128
            int a_uses = 0, rb_cur = -1;
            bool ok = true;
            SchedCursor cur(p.sc, t_begin);
            // S (and dP) of tile j into buffer j % NB, once the epilogue has read tile j - NB out of it
            auto issue_s = [&](int64_t j) -> bool {
                const int rb = cur.rb;
                cur.next(p.sc);
                if (rb != rb_cur) {
                    if (a_uses > 0) mma_commit(a_empty);  // the old row block is free once its MMAs finish
                    if (!mbar_wait(a_full, a_uses & 1, p.err, 43)) return false;
                    ++a_uses;
                    rb_cur = rb;
                }
                const int s = (int)(j % kStages), r = (int)(j / kStages), b = (int)(j % NB);
                if (j >= NB && !mbar_wait(s_free + b, (uint32_t)((j / NB - 1) & 1), p.err, 53)) return false;
                if (!mbar_wait(bs_full + s, r & 1, p.err, 44)) return false;
                fence_after_sync();
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB + (size_t)s * kStage);
                const uint32_t d = tmem + (uint32_t)(b * SH::kRegion);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ko = (uint32_t)(ks * 32);
                    mma_f16(d, desc_sw128(a0 + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), idS2, ks > 0 ? 1u : 0u);
                    mma_f16(d + 64, desc_sw128(a0 + kHalf + ko, 16, 1024), desc_sw128(b0 + ko, 16, 1024), idS, 1u);
                }
                if (SH::kDP) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t ko = (uint32_t)(ks * 32);
                        mma_f16(d + 128, desc_sw128(a0 + 2 * kHalf + ko, 16, 1024),
                                desc_sw128(b0 + 2 * kTile + ko, 16, 1024), idS2, ks > 0 ? 1u : 0u);
                        mma_f16(d + 192, desc_sw128(a0 + 3 * kHalf + ko, 16, 1024),
                                desc_sw128(b0 + 2 * kTile + ko, 16, 1024), idS, 1u);
                    }
                }
                mma_commit(s_full + b);
                return true;
            };
            // the output blocks of tile i from its kappa in TMEM. The epilogue stores kappa (w_full) only after
            // it has taken the previous tile's outputs out of the accumulators.
            auto issue_out = [&](int64_t i) -> bool {
                const int s = (int)(i % kStages);
                if (!mbar_wait(w_full, (uint32_t)(i & 1), p.err, 45)) return false;
                fence_after_sync();
                const uint32_t b0 = smem_u32(sB + (size_t)s * kStage);
#pragma unroll
                for (int o = 0; o < NO; ++o) {
                    const uint32_t kh = tmem + SH::kap(o), kl = kh + 32;
                    const uint32_t acc = tmem + SH::acc(o);
                    const uint32_t bb = b0 + SH::out_b(o);
                    // per 16 streamed points (one epilogue part): the stage's hi and lo feature blocks, MN-major
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t bo = bb + (uint32_t)(ks * 16 * kRowB);
                        if (SH::kWide) {
                            mma_f16_ta(acc, kh + (uint32_t)(ks * 8), desc_sw128(bo, kTile, 1024), idO2, ks > 0 ? 1u : 0u);
                            mma_f16_ta(acc + 64, kl + (uint32_t)(ks * 8), desc_sw128(bo, kTile, 1024), idO, 1u);
                        } else {
                            mma_f16_ta(acc, kl + (uint32_t)(ks * 8), desc_sw128(bo, kTile, 1024), idO, ks > 0 ? 1u : 0u);
                            mma_f16_ta(acc, kh + (uint32_t)(ks * 8), desc_sw128(bo + kTile, kTile, 1024), idO, 1u);
                            mma_f16_ta(acc, kh + (uint32_t)(ks * 8), desc_sw128(bo, kTile, 1024), idO, 1u);
                        }
                    }
                }
                mma_commit(bs_empty + s);  // the stage fed S, dP and the outputs
                mma_commit(o_full);
                return true;
            };
            // S (and dP) run NB tiles ahead: tile i + NB goes in as soon as the epilogue has read tile i
            for (int64_t j = 0; j < n && j < NB && ok; ++j) ok = issue_s(j);
            for (int64_t i = 0; i < n && ok; ++i) {
                if (i + NB < n) ok = issue_s(i + NB);
                if (ok) ok = issue_out(i);
            }
        }
    } else {
        // ---------------- epilogue: four warps per TMEM lane quarter; part p owns tile columns
        // [16 p, 16 p + 16) (one output K step) and output features [16 p, 16 p + 16)
        const int q = warp & 3;
        const int part = (warp - 2) >> 2;
        const int lr = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        // constants: the unscale factors of S (base 2, with the score's scale) and dP
        const int eQ = gexp(p.gmax, gQ), eK = gexp(p.gmax, gK), eV = gexp(p.gmax, gV), eD = gexp(p.gmax, gD);
        const float cS = pow2i(-eQ) * pow2i(-eK) * p.scale * kL2E;
        const float cP = pow2i(-eD) * pow2i(-eV);
        int seg = 0;
        float4 rst = make_float4(0.f, 0.f, 0.f, 0.f);
        float inv[NO];  // per output: the row's factor from the accumulator to the result
        float acc[NO][kCols];
#pragma unroll
        for (int o = 0; o < NO; ++o) {
            inv[o] = 0.f;
#pragma unroll
            for (int f = 0; f < kCols; ++f) acc[o][f] = 0.f;
        }
        // forward: the row's running maximum (base 2; the four parts of a row agree on it), the frames (maxima)
        // of the accumulator and of the pending tile's output, and this part's share of the row sum
        float fm = ninf<float>(), fm_acc = ninf<float>(), fm_pend = ninf<float>(), fl = 0.f;
        bool ok = true;
        // tile j's output MMAs have finished (its kappa is no longer read)
        auto wait_out = [&](int64_t j) -> bool {
            if (!mbar_wait(o_full, (uint32_t)(j & 1), p.err, 47)) return false;
            fence_after_sync();
            return true;
        };
        // add this part of the finished output blocks into the row accumulators
        auto add_out = [&]() {
            if constexpr (NO == 2 && !SH::kWide) {
                // both outputs' blocks with one wait
                float v0[kCols], v1[kCols];
                tmem_ld16x2(tmem + SH::acc(0) + lane_off + (uint32_t)(part * kCols),
                            tmem + SH::acc(1) + lane_off + (uint32_t)(part * kCols), v0, v1);
#pragma unroll
                for (int u = 0; u < kCols; ++u) {
                    acc[0][u] = fmaf(v0[u], inv[0], acc[0][u]);
                    acc[1][u] = fmaf(v1[u], inv[1], acc[1][u]);
                }
                return;
            }
#pragma unroll
            for (int o = 0; o < NO; ++o) {
                const uint32_t a = tmem + SH::acc(o) + lane_off + (uint32_t)(part * kCols);
                if (MODE == kFwd) {
                    // the accumulator into the current frame fm, the pending block from its own frame
                    const float fa = fm_acc == fm ? 1.f : ExpTraits<float>::bexp(fm_acc - fm);
                    const float fo = fm_pend == fm ? inv[o] : (fm_pend == ninf<float>() ? 0.f : inv[o] * ExpTraits<float>::bexp(fm_pend - fm));
                    float v[kCols], w[kCols];
                    tmem_ld16x2(a, a + 64, v, w);  // hi*hi, hi*lo + lo*hi
#pragma unroll
                    for (int u = 0; u < kCols; ++u) acc[o][u] = fmaf(v[u] + w[u], fo, acc[o][u] * fa);
                    fm_acc = fm;
                } else if (SH::kWide) {
                    float v[kCols], w[kCols];
                    tmem_ld16x2(a, a + 64, v, w);  // hi*hi, hi*lo + lo*hi
#pragma unroll
                    for (int u = 0; u < kCols; ++u) acc[o][u] = fmaf(v[u] + w[u], inv[o], acc[o][u]);
                } else {
                    float v[kCols];
                    tmem_ld16(a, v);
#pragma unroll
                    for (int u = 0; u < kCols; ++u) acc[o][u] = fmaf(v[u], inv[o], acc[o][u]);
                }
            }
        };
        int rb_cur = -1;
        const int etid = threadIdx.x - 64;  // 0 .. 32 kEpi - 1
        // Write this thread's partial of row block rb_cur. The CTA that completes the row block (the last
        // of the CTAs whose tile ranges meet it to count itself in) merges it into the outputs.
        auto write_partial = [&]() {
            const int64_t v = sched_pos(p.sc, rb_cur);
            float* o = p.part + (size_t)(v + blockIdx.x) * SH::kPartRows * kBM;
#pragma unroll
            for (int oo = 0; oo < NO; ++oo)
#pragma unroll
                for (int f = 0; f < kCols; ++f) o[(size_t)(oo * 64 + part * kCols + f) * kBM + lr] = acc[oo][f];
            if (MODE == kFwd) {
                if (part == 0) o[(size_t)SH::kF * kBM + lr] = fm;  // the accumulators are in frame fm
                o[(size_t)(SH::kF + 1 + part) * kBM + lr] = fl;
            }
            __threadfence();
            mbar_arrive(fl_bar);
            if (etid == 0) {
                int last = 0;
                if (mbar_wait(fl_bar, (uint32_t)(seg & 1), p.err, 48)) {
                    const int64_t t0 = tile_start(p.sc, v), t1 = tile_start(p.sc, v + 1) - 1;
                    const int need = cta_of_tile(p.T, p.G, t1) - cta_of_tile(p.T, p.G, t0) + 1;
                    last = atomicAdd(p.cnt + rb_cur, 1) + 1 == need;
                    __threadfence();
                }
                *sflag = last;
                mbar_arrive(dec_bar);
            }
            if (mbar_wait(dec_bar, (uint32_t)(seg & 1), p.err, 49) && *sflag) merge_row<MODE>(p, rb_cur, etid % kBM, etid / kBM);
            ++seg;
        };
        int64_t pending = -1;
        SchedCursor cur(p.sc, t_begin);
        for (int64_t i = 0; i < n && ok; ++i, cur.next(p.sc)) {
            const int rb = cur.rb, ct = cur.ct;
            if (rb != rb_cur) {
                if (pending >= 0) {
                    ok = wait_out(pending);
                    if (!ok) break;
                    add_out();
                    pending = -1;
                }
                if (rb_cur >= 0) write_partial();
                rb_cur = rb;
#pragma unroll
                for (int o = 0; o < NO; ++o)
#pragma unroll
                    for (int f = 0; f < kCols; ++f) acc[o][f] = 0.f;
                fm = fm_acc = fm_pend = ninf<float>();
                fl = 0.f;
                // row stats, padded to whole row blocks: queries (14 - lse_i log2 e, delta_i, E_i - lse_i log2 e,
                // 2^-E_i), keys (2^(E_j - 14), 2^-E_j, 0, 0)
                rst = p.rstat[(int64_t)rb * kBM + lr];
                if (MODE == kFwd) inv[0] = pow2i(-eV);  // kappa's 2^(6 - m) cancels against the row sum's
                if (MODE == kRowSweep) inv[0] = rst.w * pow2i(-eK) * p.scale;
                if (MODE == kColSweep) {
                    inv[0] = rst.y * pow2i(-eQ) * p.scale;
                    inv[NO - 1] = pow2i(-14) * pow2i(-eD);
                }
            }
            const int b = (int)(i % NB), s = (int)(i % kStages);
            ok = mbar_wait(s_full + b, (uint32_t)((i / NB) & 1), p.err, 50);
            if (ok && CST) ok = mbar_wait(bs_full + s, (uint32_t)((i / kStages) & 1), p.err, 51);  // column stats
            if (!ok) break;
            fence_after_sync();
            const float4* st = sStat + s * kBN + part * kCols;
            const uint32_t reg = tmem + lane_off + (uint32_t)(b * SH::kRegion + part * kCols);
            float k0[kCols], k1[kCols];
            if (MODE == kFwd) {
                // O: kappa = 2^(s2 - m + 6) in the row's running frame m
                float v[kCols], w[kCols];
                tmem_ld16x2(reg, reg + 64, v, w);  // S: hi*hi, hi*lo + lo*hi
                fence_before_sync();
                mbar_arrive(s_free + b);
                // kept columns of this slice (past the streamed set's end or outside a pair mask: -inf)
                const int64_t base = (int64_t)ct * kBN + part * kCols, me = (int64_t)rb * kBM + lr;
                int64_t lo = 0, hi = p.C - base;
                if (p.sc.pm == kPairsCausal) {
                    hi = min(hi, me - base + 1);
                } else if (p.sc.pm == kPairsBand) {
                    lo = me - p.sc.band - base;
                    hi = min(hi, me + p.sc.band - base + 1);
                }
                float s2[kCols], lm = ninf<float>();
#pragma unroll
                for (int u = 0; u < kCols; ++u) {
                    s2[u] = (u >= lo && u < hi) ? (v[u] + w[u]) * cS : ninf<float>();
                    lm = fmaxf(lm, s2[u]);
                }
                // the tile maximum of the row over its four parts, through shared memory (one arrival per warp)
                const int xp = (int)(i & 1);
                xm[(xp * 4 + part) * kBM + lr] = lm;
                mbar_arrive_warp(x_bar + q * 2 + xp);
                ok = mbar_wait_warp(x_bar + q * 2 + xp, (uint32_t)((i >> 1) & 1), p.err, 54);
                if (!ok) break;
                const float* xr = xm + xp * 4 * kBM + lr;
                const float tmax = fmaxf(fmaxf(xr[0], xr[kBM]), fmaxf(xr[2 * kBM], xr[3 * kBM]));
                if (tmax > fm + kLazy) {  // also the first tile with a kept pair (fm = -inf)
                    if (fm != ninf<float>()) fl *= ExpTraits<float>::bexp(fm - tmax);
                    fm = tmax;
                }
                const float sh = kKapShift - fm;
#pragma unroll
                for (int u = 0; u < kCols; ++u) {
                    k0[u] = fm == ninf<float>() ? 0.f : ExpTraits<float>::bexp(s2[u] + sh);
                    fl += k0[u];
                }
            } else {
                // P (with the row's or the column's power of two) from S, then dP
                float pr[kCols];
                {
                    float v[kCols], w[kCols];
                    tmem_ld16x2(reg, reg + 64, v, w);
#pragma unroll
                    for (int u = 0; u < kCols; ++u)
                        pr[u] = ExpTraits<float>::bexp(fmaf(v[u] + w[u], cS, MODE == kRowSweep ? rst.z : st[u].x));
                }
                float a[kCols], c[kCols];
                tmem_ld16x2(reg + 128, reg + 192, a, c);  // dP: hi*hi, hi*lo + lo*hi
                fence_before_sync();
                mbar_arrive(s_free + b);
#pragma unroll
                for (int u = 0; u < kCols; ++u) {
                    if (MODE == kRowSweep) {
                        k0[u] = pr[u] * fmaf(a[u] + c[u], cP, -rst.y);  // dS_ij 2^E_i
                    } else {
                        k1[u] = pr[u];                                          // P_ij 2^14
                        k0[u] = pr[u] * rst.x * fmaf(a[u] + c[u], cP, -st[u].y);  // dS_ij 2^E_j
                    }
                }
            }
            // Streamed points past the end (keys of the last tile) have S = 0 but their P is not 0: give
            // them no weight. The column sweep's padding queries carry -inf in place of 14 - lse2. A pair
            // mask keeps an interval of the slice's columns too: lo <= u < hi. The masked kappa is replaced,
            // not scaled (its P may exceed 1 or be infinite: lse leaves the pair out).
            {
                const int64_t base = (int64_t)ct * kBN + part * kCols;  // first streamed point of the slice
                const int64_t me = (int64_t)rb * kBM + lr;               // this thread's row point
                int64_t lo = 0, hi = kCols;
                if (MODE != kColSweep) hi = p.C - base;
                if (p.sc.pm == kPairsCausal) {
                    if (MODE == kColSweep) lo = me - base;      // queries i >= key j
                    else hi = min(hi, me - base + 1);           // keys j <= query i
                } else if (p.sc.pm == kPairsBand) {
                    lo = max(lo, me - p.sc.band - base);
                    hi = min(hi, me + p.sc.band - base + 1);
                }
                if (lo > 0 || hi < kCols) {
                    const int l = (int)min(max(lo, (int64_t)0), (int64_t)kCols);
                    const int h = (int)max(min(hi, (int64_t)kCols), (int64_t)0);
#pragma unroll
                    for (int u = 0; u < kCols; ++u) {
                        const bool keep = u >= l && u < h;
                        k0[u] = keep ? k0[u] : 0.f;
                        if (MODE == kColSweep) k1[u] = keep ? k1[u] : 0.f;
                    }
                }
            }
            // the previous tile's output MMAs have read their kappa before this tile's is stored, and the
            // epilogue takes their result out of the accumulators before it hands them over again
            if (pending >= 0) {
                ok = wait_out(pending);
                if (!ok) break;
            }
#pragma unroll
            for (int o = 0; o < NO; ++o) {
                uint32_t hw[kCols / 2], lw[kCols / 2];
#pragma unroll
                for (int k = 0; k < kCols / 2; ++k) {
                    const float x0 = o == 0 ? k0[2 * k] : k1[2 * k], x1 = o == 0 ? k0[2 * k + 1] : k1[2 * k + 1];
                    const __half2 h = __floats2half2_rn(x0, x1);
                    const float2 hf = __half22float2(h);
                    hw[k] = *reinterpret_cast<const uint32_t*>(&h);
                    lw[k] = pack_f16x2(x0 - hf.x, x1 - hf.y);
                }
                // kappa_hi of points [16 part, 16 part + 16) in columns kap + 8 part .. +8, kappa_lo 32 further
                tmem_st8(tmem + lane_off + SH::kap(o) + (uint32_t)(part * 8), hw);
                tmem_st8(tmem + lane_off + SH::kap(o) + (uint32_t)(32 + part * 8), lw);
            }
            tmem_st_wait();
            if (pending >= 0) add_out();
            fence_before_sync();
            mbar_arrive(w_full);
            pending = i;
            fm_pend = fm;
        }
        if (ok && pending >= 0) {
            ok = wait_out(pending);
            if (ok) add_out();
        }
        if (ok && rb_cur >= 0) write_partial();
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Global maxima for the powers of two and the kappa bounds: one warp per row (grid-stride), the block's
// maxima combined in shared memory, one atomicMax per block and quantity (the values are non-negative,
// so their float bits order like integers). A: max|A| into slot sa. B (optional): max|B| into sb, the
// largest row norm |B_r| into sbn. O (optional, with B): the largest |B_r . O_r| into sdel.
__global__ void __launch_bounds__(256) attn_reduce(const float* __restrict__ A, const float* __restrict__ B,
                                                   const float* __restrict__ O, int64_t rows, int* __restrict__ gm,
                                                   int sa, int sb, int sbn, int sdel) {
    griddep_wait();
    __shared__ float red[4][8];
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float ma = 0.f, mb = 0.f, mbn = 0.f, md = 0.f;
    for (int64_t r = (int64_t)blockIdx.x * 8 + wib; r < rows; r += (int64_t)gridDim.x * 8) {
        const float2 a = reinterpret_cast<const float2*>(A + r * 64)[lane];
        ma = fmaxf(ma, fmaxf(fabsf(a.x), fabsf(a.y)));
        if (B) {
            const float2 b = reinterpret_cast<const float2*>(B + r * 64)[lane];
            mb = fmaxf(mb, fmaxf(fabsf(b.x), fabsf(b.y)));
            float ss = fmaf(b.x, b.x, b.y * b.y);
            float d = 0.f;
            if (O) {
                const float2 o = reinterpret_cast<const float2*>(O + r * 64)[lane];
                d = fmaf(b.x, o.x, b.y * o.y);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                ss += __shfl_xor_sync(0xffffffffu, ss, off);
                d += __shfl_xor_sync(0xffffffffu, d, off);
            }
            mbn = fmaxf(mbn, sqrtf(ss));
            md = fmaxf(md, fabsf(d));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, off));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    }
    if (lane == 0) {
        red[0][wib] = ma;
        red[1][wib] = mb;
        red[2][wib] = mbn;
        red[3][wib] = md;
    }
    __syncthreads();
    if (threadIdx.x < 4) {
        float m = 0.f;
        for (int w = 0; w < 8; ++w) m = fmaxf(m, red[threadIdx.x][w]);
        const int slot = threadIdx.x == 0 ? sa : threadIdx.x == 1 ? sb : threadIdx.x == 2 ? sbn : sdel;
        if (slot >= 0) atomicMax(gm + slot, __float_as_int(m));
    }
}

// Pre-pass, one warp per row over rows_pad rows (two features per lane): the fp16 hi/lo split of A 2^eA
// (and B 2^eB), with the powers of two of the whole matrices (slots sa, sb), and the row's stats:
//   QUERY: (14 - lse log2 e, delta = B . O, E - lse log2 e, 2^-E) with E the power of two that brings the
//          bound |B_r| max_j |V_j| + |delta| of this row's |dP - delta| into [2^14, 2^15) (backward, B and O
//          given), (14 - lse log2 e, 0, 0, 0) otherwise; padding rows (-inf, 0, -inf, 0)
//   keys:  (2^(E - 14), 2^-E, 0, 0) with E from the bound |B_r| max_i |dO_i| + max_i |delta_i| (bounds),
//          zeros otherwise and for padding rows
// B, O, lse may be null. cnt: ncnt counters zeroed for the sweep that follows.
template <bool QUERY>
__global__ void __launch_bounds__(256) attn_split(const float* __restrict__ A, const float* __restrict__ B,
                                                  const float* __restrict__ O, const float* __restrict__ lse,
                                                  int64_t rows, int64_t rows_pad, const int* __restrict__ gm, int sa,
                                                  int sb, int bounds, __half2* __restrict__ Ah,
                                                  __half2* __restrict__ Al, __half2* __restrict__ Bh,
                                                  __half2* __restrict__ Bl, float4* __restrict__ stat,
                                                  int* __restrict__ cnt, int64_t ncnt) {
    griddep_wait();
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (lane == 0 && r < ncnt) cnt[r] = 0;
    if (r >= rows_pad) return;
    const __half2 z2 = __floats2half2_rn(0.f, 0.f);
    if (r >= rows) {
        Ah[r * 32 + lane] = z2;
        Al[r * 32 + lane] = z2;
        if (B) {
            Bh[r * 32 + lane] = z2;
            Bl[r * 32 + lane] = z2;
        }
        const float ninf = __int_as_float(0xff800000);
        if (lane == 0) stat[r] = QUERY ? make_float4(ninf, 0.f, ninf, 0.f) : make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    auto split = [&](const float* X, int slot, __half2* hi, __half2* lo) -> float2 {
        const float2 v = reinterpret_cast<const float2*>(X + r * 64)[lane];
        const float f = pow2i(f16_row_exponent(__int_as_float(__ldg(gm + slot))));
        const float a = v.x * f, b = v.y * f;
        const __half2 h = __floats2half2_rn(a, b);
        const float2 hf = __half22float2(h);
        hi[r * 32 + lane] = h;
        lo[r * 32 + lane] = __floats2half2_rn(a - hf.x, b - hf.y);
        return v;
    };
    split(A, sa, Ah, Al);
    float ss = 0.f, d = 0.f;
    if (B) {
        const float2 b = split(B, sb, Bh, Bl);
        ss = fmaf(b.x, b.x, b.y * b.y);
        if (O) {
            const float2 o = reinterpret_cast<const float2*>(O + r * 64)[lane];
            d = fmaf(b.x, o.x, b.y * o.y);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
            d += __shfl_xor_sync(0xffffffffu, d, off);
        }
    }
    if (lane != 0) return;
    if (QUERY) {
        const float l2 = lse ? lse[r] * kL2E : 0.f;  // the forward computes lse itself
        if (bounds) {
            const int E = f16_row_exponent(fmaf(sqrtf(ss), __int_as_float(__ldg(gm + gVn)), fabsf(d)));
            stat[r] = make_float4(14.f - l2, d, (float)E - l2, pow2i(-E));
        } else {
            stat[r] = make_float4(14.f - l2, 0.f, 0.f, 0.f);
        }
    } else {
        if (bounds) {
            const int E = f16_row_exponent(
                fmaf(sqrtf(ss), __int_as_float(__ldg(gm + gDn)), __int_as_float(__ldg(gm + gDelta))));
            stat[r] = make_float4(pow2i(E) * pow2i(-14), pow2i(-E), 0.f, 0.f);
        } else {
            stat[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

struct Plan {
    int64_t Npad, Mpad;
    size_t off_qh, off_ql, off_dh, off_dl, off_qst, off_kh, off_kl, off_vh, off_vl, off_kst, off_part, off_cntq,
        off_cntk, off_pfxq, off_pfxk, off_gmax, bytes;
};

static Plan plan_of(int64_t N, int64_t M, bool backward) {
    Plan pl;
    pl.Npad = (N + kBM - 1) / kBM * kBM;
    pl.Mpad = (M + kBM - 1) / kBM * kBM;
    const int64_t RBq = pl.Npad / kBM, RBk = pl.Mpad / kBM;
    const size_t qb = (size_t)pl.Npad * kRowB, kb = (size_t)pl.Mpad * kRowB;
    size_t o = 0;
    pl.off_qh = o; o += al256(qb);
    pl.off_ql = o; o += al256(qb);
    pl.off_dh = o; o += backward ? al256(qb) : 0;
    pl.off_dl = o; o += backward ? al256(qb) : 0;
    pl.off_qst = o; o += al256((size_t)pl.Npad * 16);
    pl.off_kh = o; o += al256(kb);
    pl.off_kl = o; o += al256(kb);
    pl.off_vh = o; o += al256(kb);
    pl.off_vl = o; o += al256(kb);
    pl.off_kst = o; o += al256((size_t)pl.Mpad * 16);
    // partial slots position + CTA: at most RB + G (consecutive CTA ranges never go back a position)
    size_t part = (size_t)(RBq + kGrid) * Shape<kFwd>::kPartRows * kBM * 4;
    if (backward) {
        const size_t pc = (size_t)(RBk + kGrid) * 128 * kBM * 4;
        part = part > pc ? part : pc;
    }
    pl.off_part = o; o += al256(part);
    pl.off_cntq = o; o += al256((size_t)RBq * 4);
    pl.off_cntk = o; o += al256((size_t)RBk * 4);
    pl.off_pfxq = o; o += al256((size_t)(RBq + 1) * 8);
    pl.off_pfxk = o; o += al256((size_t)(RBk + 1) * 8);
    pl.off_gmax = o; o += 256;
    pl.bytes = o;
    return pl;
}

// One sweep over R rows and C streamed points; with a pair mask (causal, band) only the column tiles that
// hold kept pairs, from the tile table built first into pfx. Returns the number of kernels launched.
template <int MODE>
static int run_sweep(const CUtensorMap (&m)[8], int64_t R, int64_t C, float scale, const float4* rstat,
                     const float4* cstat, const int* gmax, float* part, int* cnt, float* out0, float* out1, int acc0,
                     int pm, int64_t band, int64_t* pfx, int* err, const char* name, cudaStream_t s,
                     float* lse = nullptr) {
    const Sched sc = make_sched(pm, MODE == kColSweep ? 1 : 0, band, R, C, kBM, kBN, pm ? pfx : nullptr);
    int n = 0;
    if (pm) {
        launch_sched_prefix(sc, pfx, s);
        ++n;
    }
    const int64_t T = sched_total(sc);
    Params p;
    p.R = R;
    p.C = C;
    p.sc = sc;
    p.T = T;
    p.G = capped_grid((int)(T < kGrid ? T : kGrid));
    p.scale = scale;
    p.rstat = rstat;
    p.cstat = cstat;
    p.gmax = gmax;
    p.part = part;
    p.cnt = cnt;
    p.out0 = out0;
    p.out1 = out1;
    p.acc0 = acc0;
    p.lse = lse;
    p.err = err;
    cudaFuncSetAttribute(attn_tc<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    HookScope h(name, s);
    // launched early (programmatic dependent launch): its prologue overlaps the pre-pass's tail. The attention
    // kernels wait but never trigger their dependents early: with early triggers the attention step measured 1%
    // slower (the log-sum-exp kernels do trigger early: 2% faster).
    launch_pdl(attn_tc<MODE>, dim3(p.G), dim3(kThreads), kSmem, s, m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7], p);
    return n + 1;
}

static unsigned reduce_grid(int64_t rows) {
    const int64_t b = (rows + 7) / 8;
    return (unsigned)(b < 4 * kGrid ? b : 4 * kGrid);
}

}  // namespace attn
}  // namespace tc

size_t attn_tc_workspace(int64_t N, int64_t M, bool backward) { return tc::attn::plan_of(N, M, backward).bytes; }

// Forward: a.lse holds the row log-sum-exp (already computed on the stream); writes a.out. Returns the
// number of kernels launched, or -1 if a tensor map could not be encoded.
int launch_attn_fwd_tc(const AttnTcArgs& a, cudaStream_t s) {
    // one sweep writes out and lse
    using namespace tc;
    using namespace tc::attn;
    const Plan pl = plan_of(a.N, a.M, false);
    int* err = device_error_word();
    if (!err) return -3;
    char* ws = static_cast<char*>(a.ws);
    __half2* qh = reinterpret_cast<__half2*>(ws + pl.off_qh);
    __half2* ql = reinterpret_cast<__half2*>(ws + pl.off_ql);
    __half2* kh = reinterpret_cast<__half2*>(ws + pl.off_kh);
    __half2* kl = reinterpret_cast<__half2*>(ws + pl.off_kl);
    __half2* vh = reinterpret_cast<__half2*>(ws + pl.off_vh);
    __half2* vl = reinterpret_cast<__half2*>(ws + pl.off_vl);
    float4* qst = reinterpret_cast<float4*>(ws + pl.off_qst);
    float4* kst = reinterpret_cast<float4*>(ws + pl.off_kst);
    int* cntq = reinterpret_cast<int*>(ws + pl.off_cntq);
    int* gm = reinterpret_cast<int*>(ws + pl.off_gmax);
    CUtensorMap m[8];
    if (!make_map_f16(&m[0], qh, pl.Npad, kBM) || !make_map_f16(&m[1], ql, pl.Npad, kBM) ||
        !make_map_f16(&m[4], kh, pl.Mpad, kBN) || !make_map_f16(&m[5], kl, pl.Mpad, kBN) ||
        !make_map_f16(&m[6], vh, pl.Mpad, kBN) || !make_map_f16(&m[7], vl, pl.Mpad, kBN))
        return -1;
    m[2] = m[0];  // no second row operand in the forward
    m[3] = m[1];
    cudaMemsetAsync(gm, 0, kSlots * sizeof(int), s);
    {
        HookScope h("attn_reduce", s);
        launch_pdl(attn_reduce, dim3(reduce_grid(a.N)), dim3(256), 0, s, a.Q, nullptr, nullptr, a.N, gm, gQ, -1, -1,
                   -1);
    }
    {
        HookScope h("attn_reduce", s);
        launch_pdl(attn_reduce, dim3(reduce_grid(a.M)), dim3(256), 0, s, a.K, a.V, nullptr, a.M, gm, gK, gV, gVn, -1);
    }
    {
        HookScope h("attn_split", s);
        launch_pdl(attn_split<true>, dim3((unsigned)(pl.Npad / 8)), dim3(256), 0, s, a.Q, nullptr, nullptr, nullptr,
                   a.N, pl.Npad, gm, gQ, -1, 0, qh, ql, nullptr, nullptr, qst, cntq, pl.Npad / kBM);
    }
    {
        HookScope h("attn_split", s);
        launch_pdl(attn_split<false>, dim3((unsigned)(pl.Mpad / 8)), dim3(256), 0, s, a.K, a.V, nullptr, nullptr,
                   a.M, pl.Mpad, gm, gK, gV, 0, kh, kl, vh, vl, kst, nullptr, 0);
    }
    return 4 + run_sweep<kFwd>(m, a.N, a.M, (float)a.scale, qst, kst, gm, reinterpret_cast<float*>(ws + pl.off_part),
                               cntq, a.out, nullptr, 0, a.pm, a.band, reinterpret_cast<int64_t*>(ws + pl.off_pfxq),
                               err, "attn_fwd_tc", s, a.lse_out);
}

// Backward: dQ (row sweep) and dK, dV (column sweep); null outputs are not written (a sweep none of whose
// outputs is wanted does not run). With accumulate_dK the column sweep adds dK into its buffer, which
// then holds dQ from the row sweep (same points on both sides, one summed gradient). Returns the number
// of kernels launched, or -1 as above.
int launch_attn_bwd_tc(const AttnTcArgs& a, cudaStream_t s) {
    using namespace tc;
    using namespace tc::attn;
    const Plan pl = plan_of(a.N, a.M, true);
    int* err = device_error_word();
    if (!err) return -3;
    char* ws = static_cast<char*>(a.ws);
    __half2* qh = reinterpret_cast<__half2*>(ws + pl.off_qh);
    __half2* ql = reinterpret_cast<__half2*>(ws + pl.off_ql);
    __half2* dh = reinterpret_cast<__half2*>(ws + pl.off_dh);
    __half2* dl = reinterpret_cast<__half2*>(ws + pl.off_dl);
    __half2* kh = reinterpret_cast<__half2*>(ws + pl.off_kh);
    __half2* kl = reinterpret_cast<__half2*>(ws + pl.off_kl);
    __half2* vh = reinterpret_cast<__half2*>(ws + pl.off_vh);
    __half2* vl = reinterpret_cast<__half2*>(ws + pl.off_vl);
    float4* qst = reinterpret_cast<float4*>(ws + pl.off_qst);
    float4* kst = reinterpret_cast<float4*>(ws + pl.off_kst);
    int* cntq = reinterpret_cast<int*>(ws + pl.off_cntq);
    int* cntk = reinterpret_cast<int*>(ws + pl.off_cntk);
    int* gm = reinterpret_cast<int*>(ws + pl.off_gmax);
    float* part = reinterpret_cast<float*>(ws + pl.off_part);
    // row sweep maps: A = (Q, dO) in 128-row boxes, B = (K, V) in 64-row boxes; column sweep the reverse
    CUtensorMap mr[8], mc[8];
    if (!make_map_f16(&mr[0], qh, pl.Npad, kBM) || !make_map_f16(&mr[1], ql, pl.Npad, kBM) ||
        !make_map_f16(&mr[2], dh, pl.Npad, kBM) || !make_map_f16(&mr[3], dl, pl.Npad, kBM) ||
        !make_map_f16(&mr[4], kh, pl.Mpad, kBN) || !make_map_f16(&mr[5], kl, pl.Mpad, kBN) ||
        !make_map_f16(&mr[6], vh, pl.Mpad, kBN) || !make_map_f16(&mr[7], vl, pl.Mpad, kBN) ||
        !make_map_f16(&mc[0], kh, pl.Mpad, kBM) || !make_map_f16(&mc[1], kl, pl.Mpad, kBM) ||
        !make_map_f16(&mc[2], vh, pl.Mpad, kBM) || !make_map_f16(&mc[3], vl, pl.Mpad, kBM) ||
        !make_map_f16(&mc[4], qh, pl.Npad, kBN) || !make_map_f16(&mc[5], ql, pl.Npad, kBN) ||
        !make_map_f16(&mc[6], dh, pl.Npad, kBN) || !make_map_f16(&mc[7], dl, pl.Npad, kBN))
        return -1;
    cudaMemsetAsync(gm, 0, kSlots * sizeof(int), s);
    {
        HookScope h("attn_reduce", s);
        launch_pdl(attn_reduce, dim3(reduce_grid(a.N)), dim3(256), 0, s, a.Q, a.dO, a.O, a.N, gm, gQ, gD, gDn, gDelta);
    }
    {
        HookScope h("attn_reduce", s);
        launch_pdl(attn_reduce, dim3(reduce_grid(a.M)), dim3(256), 0, s, a.K, a.V, nullptr, a.M, gm, gK, gV, gVn, -1);
    }
    {
        HookScope h("attn_split", s);
        launch_pdl(attn_split<true>, dim3((unsigned)(pl.Npad / 8)), dim3(256), 0, s, a.Q, a.dO, a.O, a.lse, a.N,
                   pl.Npad, gm, gQ, gD, 1, qh, ql, dh, dl, qst, cntq, pl.Npad / kBM);
    }
    {
        HookScope h("attn_split", s);
        launch_pdl(attn_split<false>, dim3((unsigned)(pl.Mpad / 8)), dim3(256), 0, s, a.K, a.V, nullptr, nullptr,
                   a.M, pl.Mpad, gm, gK, gV, 1, kh, kl, vh, vl, kst, cntk, pl.Mpad / kBM);
    }
    int n = 4;
    if (a.dQ) {
        n += run_sweep<kRowSweep>(mr, a.N, a.M, (float)a.scale, qst, kst, gm, part, cntq, a.dQ, nullptr, 0, a.pm,
                                  a.band, reinterpret_cast<int64_t*>(ws + pl.off_pfxq), err, "attn_bwd_row_tc", s);
    }
    if (a.dK || a.dV) {
        n += run_sweep<kColSweep>(mc, a.M, a.N, (float)a.scale, kst, qst, gm, part, cntk, a.dK, a.dV, a.accumulate_dK,
                                  a.pm, a.band, reinterpret_cast<int64_t*>(ws + pl.off_pfxk), err, "attn_bwd_col_tc",
                                  s);
    }
    return n;
}

}  // namespace tp
