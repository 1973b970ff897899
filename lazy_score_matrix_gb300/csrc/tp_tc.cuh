// Blackwell (sm_103a) building blocks for the tensor-core path: inline PTX for mbarriers, TMA tile
// loads, TMEM allocation, tcgen05.mma and tcgen05.ld, and the shared-memory descriptors of the
// 128-byte-swizzled operand tiles. Every wait is bounded: past its limit it records an error code and
// returns false, so a kernel never spins forever.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tp_device.cuh"

namespace tp {
namespace tc {

constexpr unsigned long long kWaitNs = 2000000000ull;  // a wait on an mbarrier gives up after 2 s
// Site codes recorded by a wait that gives up: 1 the self-test (tp_status.cu), 11-18 lse_fwd_tc, 21-34
// lse_bwd_sym_tc, 41-54 the attention sweeps, 61-71 lse_bwd_lin_tc, 81-86 topk_tc, 91-96 lse_fwd_sym_tc.
constexpr int kSelfTestCode = 1;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// The kernel's dynamic shared memory from its first 1024-byte boundary (the repeat of the 128-byte swizzle),
// taken as an offset into the array: pointers derived from it stay shared-memory pointers to the compiler,
// so their loads and stores are shared-memory instructions (a round trip through an integer address would
// make them generic ones, which wait on the long scoreboard).
__device__ __forceinline__ unsigned char* smem_base1024(unsigned char* raw) {
    return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// One poll: true once the phase with the given parity has completed; try_wait may block for a
// hardware-chosen time first. No suspend-time hint is given: with a 20 us hint the InfoNCE and attention
// steps measured 3% slower.
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete; false after limit_ns, with `code` recorded in
// the library's device error word *err unless an earlier code is there (the first failure is kept;
// tp_device_status reads it back on the host).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, int code,
                                          unsigned long long limit_ns = kWaitNs) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) break;
    }
    atomicCAS(err, 0, code);
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One arrival per warp (the barrier counts warps): the warp synchronises, so every lane's earlier
// tcgen05 operations (after its tcgen05.fence::before_thread_sync) and memory accesses are ordered before
// lane 0's arrival. 512 per-thread arrivals on one barrier are as many serialised shared-memory atomics.
// All 32 lanes must reach the call.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
// mbar_wait whose outcome all lanes of the warp share (so that control flow stays warp-uniform).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int* err, int code) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, err, code));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Fetch a tensor map (a kernel parameter) into the descriptor cache ahead of its first TMA.
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D TMA tile load into shared memory, completing on an mbarrier. x is the innermost coordinate
// (a multiple of 32 fp32 elements here, so 128-byte aligned), y the row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
// tf32 operand split x ~ hi + lo. hi keeps the sign, exponent and top 10 mantissa bits (truncation);
// lo = x - hi is exact in fp32 but has up to 13 significant bits, one or two more than tf32 holds, and
// the MMA would truncate it toward zero, shrinking every vector by up to 2^-20 of its length in the
// same direction. Rounding lo to the nearest tf32 value here (add half a tf32 ulp to the magnitude
// bits, then clear the low 13 bits) makes that error unbiased and at most 2^-21.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }
__device__ __forceinline__ float tf32_lo(float x, float hi) {
    return __uint_as_float((__float_as_uint(x - hi) + 0x1000u) & 0xFFFFE000u);
}

__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// TMEM allocation by one whole warp; the base address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols));
}

// Shared-memory descriptor of a K-major operand tile in the 128-byte-swizzled layout: rows of 128
// bytes (32 fp32 of K), 8-row swizzle atoms of 1024 bytes stacked every 1024 bytes.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;              // leading byte offset: unused by this layout
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// Shared-memory descriptor of an MN-major operand whose MN extent spans several 128-byte-swizzled
// chunks: consecutive K rows (128 bytes of MN each) inside an 8-row atom, atoms along K every 1024
// bytes, chunks along MN every `mn_stride` bytes. kMnLboIsChunk selects which descriptor field
// carries the chunk stride (the other carries the 1024-byte atom stride).
constexpr bool kMnLboIsChunk = true;
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t mn_stride) {
    const uint32_t lbo = kMnLboIsChunk ? mn_stride : 1024u, sbo = kMnLboIsChunk ? 1024u : mn_stride;
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// (row block, column tile) of consecutive tiles t = rb * CT + ct, advanced without dividing: a 64-bit
// division per tile costs the single MMA-issuing thread (and every epilogue thread) many issue slots.
struct TileCursor {
    int rb, ct, CT;
    __device__ __forceinline__ TileCursor(int64_t t, int CT_) : rb((int)(t / CT_)), ct((int)(t % CT_)), CT(CT_) {}
    __device__ __forceinline__ void next() {
        if (++ct == CT) {
            ct = 0;
            ++rb;
        }
    }
};

// Index pair masks of the tensor-core kernels (torchpairwise guide, Score Expressions: tp.masks causal
// and band): pm 1 keeps the column points j <= i of row i, pm 2 keeps |i - j| <= band, 0 keeps all.
constexpr int kPairsCausal = 1, kPairsBand = 2;
__device__ __forceinline__ bool pair_in(int pm, int64_t band, int64_t i, int64_t j) {
    if (pm == kPairsCausal) return j <= i;
    if (pm == kPairsBand) return (i > j ? i - j : j - i) <= band;
    return true;
}

// Schedules of the sweeps. Dense: row block rb streams all CT column tiles, tile t = rb * CT + ct. Under
// an index pair mask (pair_in) row block rb streams only the tiles [c0, c1) that hold a kept pair of its
// rows (an interval: causal and band keep an interval of streamed points per row); a row block keeps at
// least one tile, so every row is written (a row that keeps no pair still gets its -inf or 0 from the
// masked tile). The row blocks are then visited in the order 0, RB-1, 1, RB-2, ... (position v holds row
// block sched_rb(v)), which pairs a short row block of a causal mask with a long one, so that no CTA's
// range is made of many short row blocks (each change of row block reloads the row operand); tiles are
// numbered position by position from pfx[v].
struct Sched {
    int pm;              // 0 dense, kPairsCausal, kPairsBand
    int col;             // 1: the rows are the score's columns (keys), the stream its rows (queries)
    int64_t band;
    int64_t R, C;        // row points, streamed points
    int lbm, lbn, CT;    // log2 of the rows per block and of the streamed points per tile; column tiles
    int64_t RB;          // row blocks
    const int64_t* pfx;  // [RB + 1] first tile of each row block (masked schedules; built by sched_prefix)
};

__host__ __device__ inline Sched make_sched(int pm, int col, int64_t band, int64_t R, int64_t C, int BM, int BN,
                                            const int64_t* pfx) {
    Sched s;
    s.pm = pm;
    s.col = col;
    s.band = band;
    s.R = R;
    s.C = C;
    s.lbm = 0;
    while ((1 << s.lbm) < BM) ++s.lbm;
    s.lbn = 0;
    while ((1 << s.lbn) < BN) ++s.lbn;
    s.CT = (int)((C + BN - 1) / BN);
    s.RB = (R + BM - 1) / BM;
    s.pfx = pfx;
    return s;
}

// Row block at position v of the schedule, and the position of row block rb.
__host__ __device__ inline int64_t sched_rb(const Sched& s, int64_t v) {
    if (!s.pm) return v;
    return (v & 1) ? s.RB - 1 - (v >> 1) : (v >> 1);
}
__host__ __device__ inline int64_t sched_pos(const Sched& s, int64_t rb) {
    if (!s.pm) return rb;
    return rb < ((s.RB + 1) >> 1) ? 2 * rb : 2 * (s.RB - 1 - rb) + 1;
}

// Column tiles [c0, c1) that row block rb (< RB) streams (BM and BN are powers of two: shifts, no division).
__host__ __device__ inline void live_tiles(const Sched& s, int64_t rb, int& c0, int& c1) {
    if (s.pm == 0) {
        c0 = 0;
        c1 = s.CT;
        return;
    }
    const int64_t r0 = rb << s.lbm, r1 = (r0 + (1 << s.lbm) < s.R ? r0 + (1 << s.lbm) : s.R) - 1;
    int64_t lo = 0, hi = s.C - 1;  // streamed points kept by some row of the block
    if (s.pm == kPairsCausal) {
        if (s.col) lo = r0;              // queries i >= key j
        else hi = hi < r1 ? hi : r1;     // keys j <= query i
    } else {
        lo = r0 - s.band > 0 ? r0 - s.band : 0;
        hi = r1 + s.band < hi ? r1 + s.band : hi;
    }
    if (lo <= hi) {  // 0 <= lo <= hi < C
        c0 = (int)(lo >> s.lbn);
        c1 = (int)(hi >> s.lbn) + 1;
    } else {  // no kept pair: one tile, fully masked
        const int64_t a = lo < s.C - 1 ? lo : s.C - 1;
        c0 = (int)(a >> s.lbn);
        c1 = c0 + 1;
    }
}

__host__ __device__ inline int64_t sched_tiles(const Sched& s, int64_t rb) {
    int c0, c1;
    live_tiles(s, rb, c0, c1);
    return c1 - c0;
}

// Tiles of the whole schedule (host: the grid and the ranges of the CTAs follow from it).
inline int64_t sched_total(const Sched& s) {
    if (!s.pm) return s.RB * s.CT;
    int64_t T = 0;
    for (int64_t rb = 0; rb < s.RB; ++rb) T += sched_tiles(s, rb);
    return T;
}

// First tile of position v (v <= RB; pfx[RB] is the tile count).
__device__ __forceinline__ int64_t tile_start(const Sched& s, int64_t v) {
    return s.pm ? __ldg(s.pfx + v) : v * s.CT;
}

// Position of tile t: the largest v with tile_start(v) <= t.
__device__ inline int64_t pos_of_tile(const Sched& s, int64_t t) {
    if (!s.pm) return t / s.CT;
    int64_t lo = 0, hi = s.RB;  // pfx[lo] <= t < pfx[hi]
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if (__ldg(s.pfx + mid) <= t) lo = mid;
        else hi = mid;
    }
    return lo;
}

// (row block, column tile) of consecutive tiles of a schedule.
struct SchedCursor {
    int64_t v;  // position
    int rb, ct, c1;
    __device__ __forceinline__ SchedCursor(const Sched& s, int64_t t) {
        v = pos_of_tile(s, t);
        rb = (int)sched_rb(s, v);
        int c0;
        live_tiles(s, rb, c0, c1);
        ct = c0 + (int)(t - tile_start(s, v));
    }
    __device__ __forceinline__ void next(const Sched& s) {
        if (++ct == c1) {
            ++v;
            if (v < s.RB) {
                rb = (int)sched_rb(s, v);
                live_tiles(s, rb, ct, c1);
            }
        }
    }
};

// Persistent schedules: the tiles t = rb * CT + ct are cut into G contiguous ranges, one per CTA.
// First tile of CTA c: floor(T c / G). 32-bit division whenever T G fits (every practical size).
__host__ __device__ inline int64_t range_start(int64_t T, int G, int c) {
    if ((unsigned long long)T * (unsigned)G < (1ull << 32)) return (int64_t)((uint32_t)T * (uint32_t)c / (uint32_t)G);
    return (T * c) / G;
}
// The CTA whose range holds tile t: the largest c with floor(T c / G) <= t, i.e. T c < G (t + 1).
__host__ __device__ inline int cta_of_tile(int64_t T, int G, int64_t t) {
    if ((unsigned long long)T * (unsigned)G < (1ull << 32))
        return (int)(((uint32_t)G * (uint32_t)(t + 1) - 1u) / (uint32_t)T);
    return (int)(((int64_t)G * (t + 1) - 1) / T);
}
// Row block of tile t (t < T).
__host__ __device__ inline int rb_of_tile(int64_t t, int CT) {
    return t < (1ll << 32) ? (int)((uint32_t)t / (uint32_t)CT) : (int)(t / CT);
}

// The upper triangle of a symmetric sweep (the log-sum-exp forward for X = Y): tiles (I, J), J >= I, of
// RB row blocks, numbered row-block major. First tile of row block I:
__host__ __device__ inline int64_t sym_start(int64_t I, int64_t RB) { return I * RB - I * (I - 1) / 2; }

// (row block, column block) of consecutive tiles of the triangle.
struct SymCursor {
    int I, J, RB;
    __host__ __device__ SymCursor(int64_t t, int RB_) : I(0), J(0), RB(RB_) {
        while (I + 1 < RB && sym_start(I + 1, RB) <= t) ++I;
        J = I + (int)(t - sym_start(I, RB));
    }
    __host__ __device__ void next() {
        if (++J == RB) {
            ++I;
            J = I;
        }
    }
};

// Pack two floats into fp16x2 (a in the low half), rounded to nearest.
__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Instruction descriptor: kind::tf32, fp32 accumulate, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor: kind::tf32, fp32 accumulate, A K-major, B MN-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32_bmn(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (1u << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D[tmem] (+)= A[tmem] * B[smem]^T (A read from tensor memory), issued by one thread.
__device__ __forceinline__ void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// kind::f16 (fp16 operands, fp32 accumulate). A and B are both fp16. A K-major; B K-major, or MN-major
// when b_mn (N contiguous in shared memory), M x N. One MMA covers K = 16 (32 bytes of a 128-byte row).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn) {
    return (1u << 4) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 128-byte-swizzled shared-memory descriptor with explicit strides: sbo is the byte distance between
// 8-row groups along the strided dimension; lbo (MN-major operands only) the byte distance between
// 64-element-wide groups along MN. For K-major operands lbo is unused.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16: A's 16 K values of a row in 8 TMEM columns, two per
// column (the lower K index in the low 16 bits).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// 2^e as a float, for e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// Exponent e that brings the largest magnitude m of a row into [2^14, 2^15) (the top of fp16's range,
// so that the lo parts of all but negligible elements stay normal), clamped so 2^e and 2^-e are normal.
__device__ __forceinline__ int f16_row_exponent(float m) {
    if (!(m > 0.f)) return 0;
    const int ex = ((__float_as_int(m) >> 23) & 0xFF) - 127;  // floor(log2 m) for normal m
    const int e = 14 - ex;
    return e < -126 ? -126 : (e > 126 ? 126 : e);
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Arrive on an mbarrier once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Two blocks of 32 consecutive fp32 columns of this thread's TMEM lane, one wait for both.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&va)[32], float (&vb)[32]) {
    uint32_t r[32], q[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta));
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]), "=r"(q[8]),
          "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15]), "=r"(q[16]),
          "=r"(q[17]), "=r"(q[18]), "=r"(q[19]), "=r"(q[20]), "=r"(q[21]), "=r"(q[22]), "=r"(q[23]), "=r"(q[24]),
          "=r"(q[25]), "=r"(q[26]), "=r"(q[27]), "=r"(q[28]), "=r"(q[29]), "=r"(q[30]), "=r"(q[31])
        : "r"(tb));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        va[u] = __uint_as_float(r[u]);
        vb[u] = __uint_as_float(q[u]);
    }
}

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape: warp w reads lanes
// 32*(w%4) .. 32*(w%4)+31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int u = 0; u < 32; ++u) v[u] = __uint_as_float(r[u]);
}

// Store 32 fp32 values into 32 consecutive columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}
// 16-column variants of the two above.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int u = 0; u < 16; ++u) v[u] = __uint_as_float(r[u]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

// 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Two 16-column loads of this thread's TMEM lane and one wait for both.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float (&va)[16], float (&vb)[16]) {
    uint32_t r[16], q[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(ta));
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]), "=r"(q[8]),
          "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15])
        : "r"(tb));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        va[u] = __uint_as_float(r[u]);
        vb[u] = __uint_as_float(q[u]);
    }
}

template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[NC]) {
    static_assert(NC == 16 || NC == 32, "16 or 32 columns");
    if constexpr (NC == 16) tmem_ld16(taddr, v);
    else tmem_ld32(taddr, v);
}
template <int NC>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float (&v)[NC]) {
    static_assert(NC == 16 || NC == 32, "16 or 32 columns");
    if constexpr (NC == 16) tmem_st16(taddr, v);
    else tmem_st32(taddr, v);
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace tp
