// Launch arguments shared by the host dispatch and the kernels (plain data, no CUDA types).
#pragma once

#include <stdint.h>

namespace tp {

constexpr int kThreads = 128;  // threads per CTA; every thread owns one point
constexpr int kTile = 32;      // streamed points per shared-memory tile

struct SweepArgs {
    const void* P;  // own points [nP, D]
    const void* Q;  // streamed points [nQ, D]
    int64_t nP, nQ;
    int D, C;
    int metric;
    double gamma, scale;
    int apply_exp;
    const void *pb, *qb, *pw, *qw;  // own/other side bias and weight, or NULL
    int affine;                     // any bias or weight present
    const void* Vq;                 // streamed value rows [nQ, VW]
    const void* Vp;                 // own value rows [nP, *]
    const void* lse;                // [rows] saved row log-sum-exp
    const void* glse;               // [rows] upstream gradient of lse
    const void* delta;              // [rows] softmax: dO_i . out_i
    int exclude_self;
    // pair mask (tp_pair_mask): 0 none, 1 causal (j <= i), 2 band (|i - j| <= band), 3 same group. The
    // sweep's own points are the rows i, or the columns j when pcol (a column sweep); pg / qg are the own
    // and the streamed side's group ids.
    int pm, pcol;
    int64_t band;
    const int *pg, *qg;
    int splits;
    int64_t cps;  // streamed points per split (multiple of kTile)
    void* out;
    void* out2;
    void* ws;
    void* gP;   // gradient of the own points [nP, D]
    void* gPb;  // own-side bias gradient [nP]
    void* gPw;  // own-side weight gradient [nP]
    void* gV;   // value gradient [nP, C] (column sweep)
    int accumulate;  // add the own-point gradient into gP instead of writing it
    int vecQ, vecV, vecVp;
    double inv_n;
    int k, largest;
};

// Tensor-core attention (fp32, D = C = 64, linear score times `scale`): out = softmax(scale Q K^T) V.
// Q [N, 64], K [M, 64], V [M, 64]; lse [N] the natural-log row log-sum-exp of the scores.
struct AttnTcArgs {
    const float *Q, *K, *V;
    int64_t N, M;
    double scale;
    const float* lse;        // backward: the forward's row log-sum-exp [N]
    const float *O, *dO;     // backward: the forward output and its upstream gradient [N, 64]
    float* out;              // forward output [N, 64]
    float* lse_out;          // forward output: the row log-sum-exp [N]
    float *dQ, *dK, *dV;     // backward outputs (null: not wanted)
    int accumulate_dK;       // add dK into its buffer (dQ and dK of the same points summed in one buffer)
    int pm;                  // pair mask: 0 none, 1 causal (j <= i), 2 band (|i - j| <= band)
    int64_t band;
    void* ws;
};

enum FwdMode : int { kMatmul = 0, kSoftmax = 1, kLse = 2, kDisp = 3, kSvgd = 4 };

// kBLseSym: logsumexp backward when X and Y are the same points and the score is symmetric (no
// row/column parameters): one sweep gives the summed gradient sum_j (H_kj + H_jk) dt_kj/dz_k.
enum BwdMode : int { kBMatmul = 0, kBSoftmax = 1, kBLse = 2, kBDisp = 3, kBLseSym = 4 };
enum Side : int { kRow = 0, kCol = 1 };


}  // namespace tp
