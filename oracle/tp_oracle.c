/*
 * Oracle for the streamed pairwise score consumers: TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct fp64 CPU loops. Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library; the product path never does. It shares no code,
 * header, helper or constant with the CUDA library.
 *
 * What is computed follows "Using Torchpairwise in Models" (torchpairwise guide, ml.html):
 *   - intro: scores S[i,j] = f(x_i, y_j) are bound lazily and consumed without storing [N,M];
 *     first derivatives replay the pairs.
 *   - "Score Expressions": per-row/per-column offsets (add_rows/add_columns), per-row/per-column
 *     weights (weight_rows/weight_columns), scalar scale and exp are folded into the score.
 *   - "Task Map": softmax_matmul(V) (attention row), K @ V (kernel attention row), row logsumexp
 *     with exclude_self (InfoNCE row), topk(k, largest=False) with exact tie order (k-NN row).
 *   - "Stein Variational Gradient Descent": the rbf kernel exp(-gamma |x-y|^2), its displacement
 *     sum_j k_ij (x_j - x_i), and the SVGD direction.
 *   - "Score Expressions" and "Task Map": pair masks tp.masks causal, band, same_group. Read here as
 *     removing the masked pairs from the consumer: no term in a sum, log-sum-exp or softmax, never
 *     selected by top-k (a row with fewer than k kept pairs pads with value +-inf and index -1), no
 *     gradient; a softmax row with no kept pair is 0.
 *
 * Score, in one fixed order (the reading adopted for the expression nodes the guide calls fused):
 *   base = |x-y|^2 (sqeuclidean) | x.y (linear) | exp(-gamma |x-y|^2) (rbf)
 *   t    = scale * wr_i * wc_j * base + br_i + bc_j      (absent weight = 1, absent bias = 0)
 *   S    = apply_exp ? exp(t) : t
 * Distances use the direct difference form, never the norm expansion. Every reduction is a plain
 * sum in fp64; logsumexp and softmax take the row maximum in a first pass and sum in a second.
 * Backward is the analytic chain rule in two loops: a row loop for dX and the per-row parameter
 * gradients, then a column loop for dY, dV and the per-column parameter gradients.
 *
 * Pins (tests/test_oracle_pins.py): dense fp64 torch brute force with torch.autograd, central
 * finite differences, and the closed forms the guide fixes (rbf(x,x) = 1, the row-mass column of
 * K @ [V | 1], softmax rows summing to 1, lse of a constant row, the SVGD formula).
 *
 * Parallelism: rows (then columns) are split over pthreads; each row or column is computed by
 * exactly one thread with the same sequential loop, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_SQEUCLIDEAN 0
#define OR_LINEAR 1
#define OR_RBF 2

#define OR_PAIRS_ALL 0
#define OR_PAIRS_CAUSAL 1     /* keep j <= i */
#define OR_PAIRS_BAND 2       /* keep |i - j| <= band */
#define OR_PAIRS_SAME_GROUP 3 /* keep row_group[i] == col_group[j] */

typedef struct {
    int metric;
    double gamma;
    double scale;
    int apply_exp;
    const double *row_bias, *col_bias, *row_weight, *col_weight; /* [N] / [M] or NULL */
    int pair_mask;
    int64_t band;
    const int32_t *row_group, *col_group; /* [N] / [M], same-group masks only */
} or_score;

/* whether the pair (i, j) stays in the consumer under the score's pair mask */
static int pair_kept(const or_score *s, int64_t i, int64_t j) {
    switch (s->pair_mask) {
    case OR_PAIRS_CAUSAL: return j <= i;
    case OR_PAIRS_BAND: return llabs(i - j) <= s->band;
    case OR_PAIRS_SAME_GROUP: return s->row_group[i] == s->col_group[j];
    default: return 1;
    }
}

typedef struct {
    const double *X, *Y; /* [N,D], [M,D] row-major */
    int64_t N, M, D;
} or_pairs;

/* ------------------------------------------------------------------------------------------ */
/* parallel for                                                                               */
/* ------------------------------------------------------------------------------------------ */

typedef void (*or_body)(void *ctx, int64_t idx);

typedef struct {
    or_body body;
    void *ctx;
    int64_t n;
    int64_t next;
    pthread_mutex_t lock;
} or_pool;

static void *or_worker(void *arg) {
    or_pool *p = (or_pool *)arg;
    for (;;) {
        int64_t lo, hi;
        pthread_mutex_lock(&p->lock);
        lo = p->next;
        hi = lo + 16 < p->n ? lo + 16 : p->n;
        p->next = hi;
        pthread_mutex_unlock(&p->lock);
        if (lo >= p->n) break;
        for (int64_t i = lo; i < hi; ++i) p->body(p->ctx, i);
    }
    return NULL;
}

int or_hardware_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int g_threads = 0; /* 0 = all online cores */

void or_set_threads(int n) { g_threads = n; }

int or_get_threads(void) { return g_threads > 0 ? g_threads : or_hardware_threads(); }

static void or_parallel_for(int64_t n, or_body body, void *ctx) {
    int nt = or_get_threads();
    if (nt > 256) nt = 256;
    if (n <= 0) return;
    if (nt <= 1 || n < 2) {
        for (int64_t i = 0; i < n; ++i) body(ctx, i);
        return;
    }
    or_pool p;
    p.body = body;
    p.ctx = ctx;
    p.n = n;
    p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nt; ++t)
        if (pthread_create(&th[t], NULL, or_worker, &p) == 0) ++started;
    if (started == 0) or_worker(&p);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&p.lock);
}

/* ------------------------------------------------------------------------------------------ */
/* score and its partial derivatives                                                          */
/* ------------------------------------------------------------------------------------------ */

static double row_w(const or_score *s, int64_t i) { return s->row_weight ? s->row_weight[i] : 1.0; }
static double col_w(const or_score *s, int64_t j) { return s->col_weight ? s->col_weight[j] : 1.0; }
static double row_b(const or_score *s, int64_t i) { return s->row_bias ? s->row_bias[i] : 0.0; }
static double col_b(const or_score *s, int64_t j) { return s->col_bias ? s->col_bias[j] : 0.0; }

/* base score of one pair, from the metric's definition */
static double base_of(const or_score *s, const double *x, const double *y, int64_t D) {
    double acc = 0.0;
    if (s->metric == OR_LINEAR) {
        for (int64_t d = 0; d < D; ++d) acc += x[d] * y[d];
        return acc;
    }
    for (int64_t d = 0; d < D; ++d) {
        double diff = x[d] - y[d];
        acc += diff * diff;
    }
    if (s->metric == OR_RBF) return exp(-s->gamma * acc);
    return acc;
}

typedef struct {
    double base; /* metric value */
    double t;    /* score before the optional exp */
    double S;    /* final score */
} or_pair_val;

static or_pair_val pair_eval(const or_score *s, const or_pairs *p, int64_t i, int64_t j) {
    or_pair_val v;
    const double *x = p->X + i * p->D, *y = p->Y + j * p->D;
    v.base = base_of(s, x, y, p->D);
    v.t = s->scale * row_w(s, i) * col_w(s, j) * v.base + row_b(s, i) + col_b(s, j);
    v.S = s->apply_exp ? exp(v.t) : v.t;
    return v;
}

/*
 * Given G = dL/dS for pair (i,j), add the chain-rule terms into
 *   gx[D] (dL/dx_i) when gx != NULL, gy[D] (dL/dy_j) when gy != NULL,
 *   *gbr, *gwr (row bias / weight), *gbc, *gwc (column bias / weight) when non-NULL.
 */
static void pair_chain(const or_score *s, const or_pairs *p, int64_t i, int64_t j, or_pair_val v,
                       double G, double *gx, double *gy, double *gbr, double *gwr, double *gbc,
                       double *gwc) {
    const double *x = p->X + i * p->D, *y = p->Y + j * p->D;
    double H = s->apply_exp ? G * v.S : G; /* dL/dt */
    if (gbr) *gbr += H;
    if (gbc) *gbc += H;
    if (gwr) *gwr += H * s->scale * col_w(s, j) * v.base;
    if (gwc) *gwc += H * s->scale * row_w(s, i) * v.base;
    double E = H * s->scale * row_w(s, i) * col_w(s, j); /* dL/dbase */
    for (int64_t d = 0; d < p->D; ++d) {
        double dbx, dby; /* dbase/dx_id, dbase/dy_jd */
        if (s->metric == OR_LINEAR) {
            dbx = y[d];
            dby = x[d];
        } else if (s->metric == OR_SQEUCLIDEAN) {
            dbx = 2.0 * (x[d] - y[d]);
            dby = -2.0 * (x[d] - y[d]);
        } else {
            dbx = -2.0 * s->gamma * v.base * (x[d] - y[d]);
            dby = 2.0 * s->gamma * v.base * (x[d] - y[d]);
        }
        if (gx) gx[d] += E * dbx;
        if (gy) gy[d] += E * dby;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* forward consumers                                                                          */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    const or_pairs *p;
    const or_score *s;
    const double *V;
    int64_t C;
    double *out;
    double *out2;
    int exclude_self;
    int k, largest;
    int64_t *idx;
    volatile int failed;
    const double *aux0, *aux1, *aux2, *aux3;
    double *g0, *g1, *g2, *g3, *g4;
} or_ctx;

/* K @ V: out_i = sum_j S_ij V_j  ("Task Map", kernel attention row) */
static void matmul_row(void *c_, int64_t i) {
    or_ctx *c = (or_ctx *)c_;
    double *o = c->out + i * c->C;
    for (int64_t cc = 0; cc < c->C; ++cc) o[cc] = 0.0;
    for (int64_t j = 0; j < c->p->M; ++j) {
        if (!pair_kept(c->s, i, j)) continue;
        double S = pair_eval(c->s, c->p, i, j).S;
        for (int64_t cc = 0; cc < c->C; ++cc) o[cc] += S * c->V[j * c->C + cc];
    }
}

int or_matmul(const or_pairs *p, const or_score *s, const double *V, int64_t C, double *out) {
    or_ctx c = {0};
    c.p = p; c.s = s; c.V = V; c.C = C; c.out = out;
    or_parallel_for(p->N, matmul_row, &c);
    return 0;
}

/* two-pass row logsumexp: max first, then the shifted sum; -inf for an empty row */
static double row_lse(const or_score *s, const or_pairs *p, int64_t i, int exclude_self) {
    double m = -INFINITY;
    for (int64_t j = 0; j < p->M; ++j) {
        if ((exclude_self && j == i) || !pair_kept(s, i, j)) continue;
        double S = pair_eval(s, p, i, j).S;
        if (S > m) m = S;
    }
    if (m == -INFINITY) return -INFINITY;
    double sum = 0.0;
    for (int64_t j = 0; j < p->M; ++j) {
        if ((exclude_self && j == i) || !pair_kept(s, i, j)) continue;
        sum += exp(pair_eval(s, p, i, j).S - m);
    }
    return m + log(sum);
}

/* lse_i = log sum_{j (!= i)} exp S_ij  ("Task Map", InfoNCE row; "Score Expressions" example) */
static void lse_row(void *c_, int64_t i) {
    or_ctx *c = (or_ctx *)c_;
    c->out[i] = row_lse(c->s, c->p, i, c->exclude_self);
}

int or_logsumexp(const or_pairs *p, const or_score *s, int exclude_self, double *lse) {
    if (exclude_self && p->N > p->M) return 1; /* pair (i, i) must exist for every row */
    or_ctx c = {0};
    c.p = p; c.s = s; c.out = lse; c.exclude_self = exclude_self;
    or_parallel_for(p->N, lse_row, &c);
    return 0;
}

/* out_i = sum_j softmax_j(S_ij) V_j, lse_i saved  (intro example and "Task Map" attention row) */
static void softmax_row(void *c_, int64_t i) {
    or_ctx *c = (or_ctx *)c_;
    double l = row_lse(c->s, c->p, i, 0);
    double *o = c->out + i * c->C;
    for (int64_t cc = 0; cc < c->C; ++cc) o[cc] = 0.0;
    for (int64_t j = 0; j < c->p->M && l > -INFINITY; ++j) {
        if (!pair_kept(c->s, i, j)) continue;
        double P = exp(pair_eval(c->s, c->p, i, j).S - l);
        for (int64_t cc = 0; cc < c->C; ++cc) o[cc] += P * c->V[j * c->C + cc];
    }
    if (c->out2) c->out2[i] = l;
}

int or_softmax_matmul(const or_pairs *p, const or_score *s, const double *V, int64_t C,
                      double *out, double *lse) {
    or_ctx c = {0};
    c.p = p; c.s = s; c.V = V; c.C = C; c.out = out; c.out2 = lse;
    or_parallel_for(p->N, softmax_row, &c);
    return 0;
}

/* disp_i = sum_j S_ij (y_j - x_i)  ("Stein Variational Gradient Descent", displacement method) */
static void disp_row(void *c_, int64_t i) {
    or_ctx *c = (or_ctx *)c_;
    const or_pairs *p = c->p;
    double *o = c->out + i * p->D;
    for (int64_t d = 0; d < p->D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < p->M; ++j) {
        if (!pair_kept(c->s, i, j)) continue;
        double S = pair_eval(c->s, p, i, j).S;
        for (int64_t d = 0; d < p->D; ++d) o[d] += S * (p->Y[j * p->D + d] - p->X[i * p->D + d]);
    }
}

int or_displacement(const or_pairs *p, const or_score *s, double *out) {
    or_ctx c = {0};
    c.p = p; c.s = s; c.out = out;
    or_parallel_for(p->N, disp_row, &c);
    return 0;
}

/*
 * SVGD direction, from the formula in "Stein Variational Gradient Descent":
 *   phi_i = (1/n) sum_j [ k(x_j, x_i) score_j + grad_{x_j} k(x_j, x_i) ]
 * with k the rbf kernel exp(-gamma |x_j - x_i|^2), whose gradient in x_j is
 *   -2 gamma (x_j - x_i) k(x_j, x_i).  Here X = Y = x, n = M, score is [M,D].
 * The score's scale/bias/weight/exp fields are not used: the formula is the bare rbf kernel.
 */
static void svgd_row(void *c_, int64_t i) {
    or_ctx *c = (or_ctx *)c_;
    const or_pairs *p = c->p;
    const double g = c->s->gamma;
    double *o = c->out + i * p->D;
    for (int64_t d = 0; d < p->D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < p->M; ++j) {
        const double *xj = p->Y + j * p->D, *xi = p->X + i * p->D;
        double r2 = 0.0;
        for (int64_t d = 0; d < p->D; ++d) r2 += (xj[d] - xi[d]) * (xj[d] - xi[d]);
        double k = exp(-g * r2);
        for (int64_t d = 0; d < p->D; ++d)
            o[d] += k * c->V[j * p->D + d] + (-2.0 * g * (xj[d] - xi[d]) * k);
    }
    for (int64_t d = 0; d < p->D; ++d) o[d] /= (double)p->M;
}

int or_svgd_direction(const or_pairs *p, double gamma, const double *score, double *phi) {
    or_score s;
    memset(&s, 0, sizeof s);
    s.metric = OR_RBF;
    s.gamma = gamma;
    s.scale = 1.0;
    or_ctx c = {0};
    c.p = p; c.s = &s; c.V = score; c.out = phi;
    or_parallel_for(p->N, svgd_row, &c);
    return 0;
}

/* top-k: full sort of (key, j) per row; key = S (smallest first) or -S (largest first); ties by
 * ascending index ("Task Map", k-NN row: exact tie order) */
typedef struct {
    double key;
    int64_t j;
} or_kv;

static int kv_cmp(const void *a_, const void *b_) {
    const or_kv *a = (const or_kv *)a_, *b = (const or_kv *)b_;
    if (a->key < b->key) return -1;
    if (a->key > b->key) return 1;
    return (a->j > b->j) - (a->j < b->j);
}

static void topk_row(void *c_, int64_t i) {
    or_ctx *c = (or_ctx *)c_;
    const or_pairs *p = c->p;
    or_kv *buf = (or_kv *)malloc(sizeof(or_kv) * (size_t)p->M);
    if (!buf) { /* out of host memory: the caller sees the flag */
        c->failed = 1;
        return;
    }
    int64_t n = 0;
    for (int64_t j = 0; j < p->M; ++j) {
        if (!pair_kept(c->s, i, j)) continue;
        double S = pair_eval(c->s, p, i, j).S;
        buf[n].key = c->largest ? -S : S;
        buf[n].j = j;
        ++n;
    }
    qsort(buf, (size_t)n, sizeof(or_kv), kv_cmp);
    for (int t = 0; t < c->k; ++t) {
        if (t < n) {
            c->out[i * c->k + t] = c->largest ? -buf[t].key : buf[t].key;
            c->idx[i * c->k + t] = buf[t].j;
        } else { /* fewer kept pairs than k */
            c->out[i * c->k + t] = c->largest ? -INFINITY : INFINITY;
            c->idx[i * c->k + t] = -1;
        }
    }
    free(buf);
}

int or_topk(const or_pairs *p, const or_score *s, int k, int largest, double *values,
            int64_t *indices) {
    if (k < 1 || k > p->M) return 1;
    or_ctx c = {0};
    c.p = p; c.s = s; c.k = k; c.largest = largest; c.out = values; c.idx = indices;
    or_parallel_for(p->N, topk_row, &c);
    return c.failed ? 2 : 0;
}

/* ------------------------------------------------------------------------------------------ */
/* backward: analytic chain rule, row loop then column loop                                   */
/* ------------------------------------------------------------------------------------------ */

/* consumer kinds for the shared backward driver */
#define OR_K_MATMUL 0
#define OR_K_LSE 1
#define OR_K_SOFTMAX 2
#define OR_K_DISP 3

typedef struct {
    const or_pairs *p;
    const or_score *s;
    int kind;
    int exclude_self;
    const double *V; /* [M,C] */
    int64_t C;
    const double *gout;  /* matmul/softmax: [N,C]; lse: [N]; disp: [N,D] */
    const double *lse;   /* [N] (lse, softmax) */
    const double *delta; /* [N] softmax: dO_i . out_i */
    double *dX, *dY, *dV, *dbr, *dbc, *dwr, *dwc;
} or_bwd;

/* G = dL/dS_ij for the consumer */
static double consumer_G(const or_bwd *b, int64_t i, int64_t j, double S) {
    switch (b->kind) {
    case OR_K_MATMUL: {
        double g = 0.0;
        for (int64_t c = 0; c < b->C; ++c) g += b->gout[i * b->C + c] * b->V[j * b->C + c];
        return g;
    }
    case OR_K_LSE:
        if (b->exclude_self && i == j) return 0.0;
        if (b->lse[i] == -INFINITY) return 0.0;
        return b->gout[i] * exp(S - b->lse[i]);
    case OR_K_SOFTMAX: {
        double dp = 0.0;
        for (int64_t c = 0; c < b->C; ++c) dp += b->gout[i * b->C + c] * b->V[j * b->C + c];
        return exp(S - b->lse[i]) * (dp - b->delta[i]);
    }
    default: { /* displacement: out_i = sum_j S_ij (y_j - x_i) */
        const or_pairs *p = b->p;
        double g = 0.0;
        for (int64_t d = 0; d < p->D; ++d)
            g += b->gout[i * p->D + d] * (p->Y[j * p->D + d] - p->X[i * p->D + d]);
        return g;
    }
    }
}

static void bwd_row(void *b_, int64_t i) {
    or_bwd *b = (or_bwd *)b_;
    const or_pairs *p = b->p;
    double *gx = b->dX ? b->dX + i * p->D : NULL;
    double gbr = 0.0, gwr = 0.0;
    if (gx)
        for (int64_t d = 0; d < p->D; ++d) gx[d] = 0.0;
    for (int64_t j = 0; j < p->M; ++j) {
        if (!pair_kept(b->s, i, j)) continue;
        or_pair_val v = pair_eval(b->s, p, i, j);
        double G = consumer_G(b, i, j, v.S);
        pair_chain(b->s, p, i, j, v, G, gx, NULL, &gbr, &gwr, NULL, NULL);
        if (b->kind == OR_K_DISP && gx) /* d/dx_i of S_ij (y_j - x_i) beyond S: -S_ij dO_i */
            for (int64_t d = 0; d < p->D; ++d) gx[d] -= v.S * b->gout[i * p->D + d];
    }
    if (b->dbr) b->dbr[i] = gbr;
    if (b->dwr) b->dwr[i] = gwr;
}

static void bwd_col(void *b_, int64_t j) {
    or_bwd *b = (or_bwd *)b_;
    const or_pairs *p = b->p;
    double *gy = b->dY ? b->dY + j * p->D : NULL;
    double *gv = b->dV ? b->dV + j * b->C : NULL;
    double gbc = 0.0, gwc = 0.0;
    if (gy)
        for (int64_t d = 0; d < p->D; ++d) gy[d] = 0.0;
    if (gv)
        for (int64_t c = 0; c < b->C; ++c) gv[c] = 0.0;
    for (int64_t i = 0; i < p->N; ++i) {
        if (!pair_kept(b->s, i, j)) continue;
        or_pair_val v = pair_eval(b->s, p, i, j);
        double G = consumer_G(b, i, j, v.S);
        pair_chain(b->s, p, i, j, v, G, NULL, gy, NULL, NULL, &gbc, &gwc);
        if (b->kind == OR_K_DISP && gy) /* d/dy_j of S_ij (y_j - x_i) beyond S: +S_ij dO_i */
            for (int64_t d = 0; d < p->D; ++d) gy[d] += v.S * b->gout[i * p->D + d];
        if (gv) {
            /* matmul: out_i = sum_j S_ij V_j; softmax: out_i = sum_j P_ij V_j */
            double w = v.S;
            if (b->kind == OR_K_SOFTMAX) w = exp(v.S - b->lse[i]);
            for (int64_t c = 0; c < b->C; ++c) gv[c] += w * b->gout[i * b->C + c];
        }
    }
    if (b->dbc) b->dbc[j] = gbc;
    if (b->dwc) b->dwc[j] = gwc;
}

static int run_bwd(or_bwd *b) {
    const or_pairs *p = b->p;
    int need_row = b->dX || b->dbr || b->dwr;
    int need_col = b->dY || b->dV || b->dbc || b->dwc;
    if (need_row) or_parallel_for(p->N, bwd_row, b);
    if (need_col) or_parallel_for(p->M, bwd_col, b);
    return 0;
}

int or_matmul_backward(const or_pairs *p, const or_score *s, const double *V, int64_t C,
                       const double *grad_out, double *dX, double *dY, double *dV, double *dbr,
                       double *dbc, double *dwr, double *dwc) {
    or_bwd b;
    memset(&b, 0, sizeof b);
    b.p = p; b.s = s; b.kind = OR_K_MATMUL; b.V = V; b.C = C; b.gout = grad_out;
    b.dX = dX; b.dY = dY; b.dV = dV; b.dbr = dbr; b.dbc = dbc; b.dwr = dwr; b.dwc = dwc;
    return run_bwd(&b);
}

int or_logsumexp_backward(const or_pairs *p, const or_score *s, int exclude_self,
                          const double *lse, const double *grad_lse, double *dX, double *dY,
                          double *dbr, double *dbc, double *dwr, double *dwc) {
    if (exclude_self && p->N > p->M) return 1; /* pair (i, i) must exist for every row */
    or_bwd b;
    memset(&b, 0, sizeof b);
    b.p = p; b.s = s; b.kind = OR_K_LSE; b.exclude_self = exclude_self; b.lse = lse;
    b.gout = grad_lse;
    b.dX = dX; b.dY = dY; b.dbr = dbr; b.dbc = dbc; b.dwr = dwr; b.dwc = dwc;
    return run_bwd(&b);
}

/* delta_i = dO_i . out_i, the row term of the softmax Jacobian */
static void softmax_delta_row(void *c_, int64_t i) {
    or_ctx *c = (or_ctx *)c_;
    double acc = 0.0;
    for (int64_t cc = 0; cc < c->C; ++cc) acc += c->aux0[i * c->C + cc] * c->aux1[i * c->C + cc];
    c->out[i] = acc;
}

int or_softmax_matmul_backward(const or_pairs *p, const or_score *s, const double *V, int64_t C,
                               const double *out, const double *lse, const double *grad_out,
                               double *dX, double *dY, double *dV, double *dbr, double *dbc,
                               double *dwr, double *dwc) {
    double *delta = (double *)malloc(sizeof(double) * (size_t)(p->N > 0 ? p->N : 1));
    if (!delta) return 2;
    or_ctx c = {0};
    c.C = C; c.aux0 = grad_out; c.aux1 = out; c.out = delta;
    or_parallel_for(p->N, softmax_delta_row, &c);
    or_bwd b;
    memset(&b, 0, sizeof b);
    b.p = p; b.s = s; b.kind = OR_K_SOFTMAX; b.V = V; b.C = C; b.gout = grad_out; b.lse = lse;
    b.delta = delta;
    b.dX = dX; b.dY = dY; b.dV = dV; b.dbr = dbr; b.dbc = dbc; b.dwr = dwr; b.dwc = dwc;
    int rc = run_bwd(&b);
    free(delta);
    return rc;
}

int or_displacement_backward(const or_pairs *p, const or_score *s, const double *grad_out,
                             double *dX, double *dY, double *dbr, double *dbc, double *dwr,
                             double *dwc) {
    or_bwd b;
    memset(&b, 0, sizeof b);
    b.p = p; b.s = s; b.kind = OR_K_DISP; b.gout = grad_out;
    b.dX = dX; b.dY = dY; b.dbr = dbr; b.dbc = dbc; b.dwr = dwr; b.dwc = dwc;
    return run_bwd(&b);
}

/*
 * top-k backward: gradients flow through the selected pairs only ("What to Check", gradients of
 * selections). grad_values [N,k] is dL/dS at (i, indices[i,t]). Sequential: plain and small.
 */
int or_topk_backward(const or_pairs *p, const or_score *s, int k, const int64_t *indices,
                     const double *grad_values, double *dX, double *dY, double *dbr, double *dbc,
                     double *dwr, double *dwc) {
    if (dX) memset(dX, 0, sizeof(double) * (size_t)(p->N * p->D));
    if (dY) memset(dY, 0, sizeof(double) * (size_t)(p->M * p->D));
    if (dbr) memset(dbr, 0, sizeof(double) * (size_t)p->N);
    if (dwr) memset(dwr, 0, sizeof(double) * (size_t)p->N);
    if (dbc) memset(dbc, 0, sizeof(double) * (size_t)p->M);
    if (dwc) memset(dwc, 0, sizeof(double) * (size_t)p->M);
    for (int64_t i = 0; i < p->N; ++i) {
        for (int t = 0; t < k; ++t) {
            int64_t j = indices[i * k + t];
            if (j == -1) continue; /* a padding place (fewer kept pairs than k): no gradient */
            if (j < 0 || j >= p->M) return 1;
            or_pair_val v = pair_eval(s, p, i, j);
            pair_chain(s, p, i, j, v, grad_values[i * k + t], dX ? dX + i * p->D : NULL,
                       dY ? dY + j * p->D : NULL, dbr ? dbr + i : NULL, dwr ? dwr + i : NULL,
                       dbc ? dbc + j : NULL, dwc ? dwc + j : NULL);
        }
    }
    return 0;
}

/* scalar score of one pair, exposed for pins */
double or_pair_score(const or_pairs *p, const or_score *s, int64_t i, int64_t j) {
    return pair_eval(s, p, i, j).S;
}
