/*
 * dflash_oracle.c: plain, slow CPU reference of the DFlash2 low-rank candidate selector.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU
 * baseline use this file. The product library never links it, calls it or shares code
 * with it.
 *
 * Source. The page "vllm.models.beam.nvidia.dflash2" (DFlash2 draft model for Beam
 * targets):
 *   - class DFlash2BeamCandidateSelector, its docstring and forward():
 *       the edge score of block position p, candidate c and predecessor q is the
 *       candidate's own logit plus <predecessor[q] * h_p, successor[c]>. h_p is the
 *       drafter hidden state projected to the codebook rank. The predecessor of the
 *       first position is the anchor token. Output layout:
 *       [requests, steps, top_k (predecessor), top_k].
 *   - DFlash2BeamCandidateSelector.__init__: predecessor_codebook and
 *       successor_codebook are [vocab, rank]; hidden_projection is a bias-free
 *       linear map hidden_size -> rank in params_dtype (bf16).
 *   - DFlash2BeamForCausalLM.compute_candidates: the selector's top-k candidate ids
 *       and their logits at each position.
 *
 * Readings where the page is silent:
 *   - Top-k order: logit descending; equal logits go to the lower token id; -0 and +0
 *     are equal. A NaN with the sign bit clear ranks above +inf, and one with the sign
 *     bit set ranks below -inf. NaNs of one sign are equal to each other.
 *   - unary = the selected logit itself, in fp32. With the logits processor's options
 *     (DFlash2BeamForCausalLM.__init__ on the second page: LogitsProcessor(soft_cap,
 *     scale=output_multiplier)), unary = scale * cap * tanh(x / cap), the cap applied
 *     first. The selection and order still use the raw logits: the map is strictly
 *     increasing for scale > 0.
 *   - Projection: an exact (fp64) dot product, rounded once to bf16, nearest-even.
 *   - Edges: exact (fp64) sums over the bf16 values, stored as fp32. pred*h is not
 *     rounded before the dot product.
 *
 *   - Best path over the edge scores (what consumes E is not shown on the pages; the
 *       reading is the max-sum path through the candidate lattice): for each request,
 *       one candidate per step maximising the sum of E[r,p,c_{p-1},c_p], in fp32 with
 *       the order and tie rule written at oracle_best_path below.
 *
 * Every computation is the plain definition. Top-k fully sorts the row. The dot
 * products are single fp64 loops. Rows are split across pthreads only for wall time;
 * each row is computed exactly as in the serial loop.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 helpers */

/* bf16 bit pattern -> double (exact: bf16 is the top half of an IEEE binary32). */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even, in one step (no detour through
 * binary32, which would round twice). bf16 has 8 significant bits and binary32's
 * exponent range, subnormals included. */
uint16_t oracle_bf16_round(double x) {
    if (isnan(x)) return signbit(x) ? 0xFFC0u : 0x7FC0u;
    if (isinf(x)) return signbit(x) ? 0xFF80u : 0x7F80u;
    if (x == 0.0) return signbit(x) ? 0x8000u : 0x0000u;
    int e;
    frexp(fabs(x), &e);                 /* |x| in [2^(e-1), 2^e) */
    int E = e - 1;                      /* binary exponent of |x| */
    if (E < -126) E = -126;             /* below the normal range the spacing stays 2^-133 */
    double ulp = ldexp(1.0, E - 7);     /* spacing of bf16 values near x */
    double q = nearbyint(x / ulp);      /* default rounding mode: nearest, ties to even */
    double y = q * ulp;
    if (fabs(y) >= ldexp(1.0, 128)) return signbit(x) ? 0xFF80u : 0x7F80u;
    float f = (float)y;                 /* exact: y has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- thread pool */

typedef void (*row_fn)(void* ctx, int64_t row);

typedef struct {
    row_fn fn;
    void* ctx;
    int64_t lo, hi;
} span_t;

static void* run_span(void* arg) {
    span_t* s = (span_t*)arg;
    for (int64_t r = s->lo; r < s->hi; ++r) s->fn(s->ctx, r);
    return NULL;
}

/* Call fn(ctx, r) for r in [0, rows) on `threads` threads, in contiguous spans. */
static int parallel_rows(row_fn fn, void* ctx, int64_t rows, int threads) {
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if ((int64_t)threads > rows) threads = (int)(rows > 0 ? rows : 1);
    if (threads == 1) {
        for (int64_t r = 0; r < rows; ++r) fn(ctx, r);
        return 0;
    }
    pthread_t tid[256];
    span_t span[256];
    int created[256];
    for (int t = 0; t < threads; ++t) {
        span[t].fn = fn;
        span[t].ctx = ctx;
        span[t].lo = rows * t / threads;
        span[t].hi = rows * (t + 1) / threads;
        created[t] = pthread_create(&tid[t], NULL, run_span, &span[t]) == 0;
        if (!created[t]) run_span(&span[t]);   /* no thread: run the span here */
    }
    for (int t = 0; t < threads; ++t)
        if (created[t]) pthread_join(tid[t], NULL);
    return 0;
}

/* ---------------------------------------------------------------- step 1: top-k */

typedef struct {
    float v;
    int32_t id;
} entry_t;

/* 2 for NaN with the sign clear, 0 for NaN with the sign set, 1 for any other value. */
static int nan_class(float v) {
    if (isnan(v)) return signbit(v) ? 0 : 2;
    return 1;
}

/* qsort comparator: negative when a comes first in the candidate order. */
static int entry_order(const void* pa, const void* pb) {
    const entry_t* a = (const entry_t*)pa;
    const entry_t* b = (const entry_t*)pb;
    int ca = nan_class(a->v), cb = nan_class(b->v);
    if (ca != cb) return ca > cb ? -1 : 1;
    if (ca == 1 && a->v != b->v) return a->v > b->v ? -1 : 1;   /* -0 == +0 here */
    return (a->id < b->id) ? -1 : (a->id > b->id ? 1 : 0);
}

typedef struct {
    const float* logits;
    int64_t V;
    int K;
    double softcap;   /* <= 0: no cap */
    double scale;
    int32_t* ids;
    float* unary;
    int failed;
} topk_ctx;

/* The logits processor applied to one selected logit: cap * tanh(x / cap), then * scale. */
static float processed_logit(float x, double softcap, double scale) {
    double v = (double)x;
    if (softcap > 0.0) v = softcap * tanh(v / softcap);
    return (float)(v * scale);
}

static void topk_row(void* vctx, int64_t r) {
    topk_ctx* c = (topk_ctx*)vctx;
    entry_t* e = (entry_t*)malloc((size_t)c->V * sizeof(entry_t));
    if (!e) {
        c->failed = 1;
        return;
    }
    const float* row = c->logits + r * c->V;
    for (int64_t v = 0; v < c->V; ++v) {
        e[v].v = row[v];
        e[v].id = (int32_t)v;
    }
    qsort(e, (size_t)c->V, sizeof(entry_t), entry_order);
    for (int k = 0; k < c->K; ++k) {
        c->ids[r * c->K + k] = e[k].id;
        c->unary[r * c->K + k] = processed_logit(e[k].v, c->softcap, c->scale);
    }
    free(e);
}

/* For each of `rows` rows of `V` logits: the K first tokens of the candidate order
 * (logit descending, then token id ascending) and their processed logits (softcap <= 0
 * and scale = 1 leave them raw). Returns 0, or -1 on bad arguments or allocation failure. */
int oracle_topk(const float* logits, int64_t rows, int64_t V, int K, double softcap,
                double scale, int32_t* ids, float* unary, int threads) {
    if (!logits || !ids || !unary || rows < 0 || V < 1 || K < 1 || K > V) return -1;
    if (!(scale > 0.0)) return -1;
    topk_ctx c = {logits, V, K, softcap, scale, ids, unary, 0};
    parallel_rows(topk_row, &c, rows, threads);
    return c.failed ? -1 : 0;
}

/* ---------------------------------------------------------------- candidate head from the LM head */

typedef struct {
    const uint16_t* hidden;   /* [rows, H] bf16 bits */
    const uint16_t* lm_head;  /* [V, H] bf16 bits */
    int64_t H, V;
    int K;
    double softcap, scale;
    int32_t* ids;
    float* unary;
    double* logits_out;       /* [rows, V] exact logits, or NULL */
    int failed;
} lmhead_ctx;

/* Order of (exact logit, id): the candidate order of the top-k, on fp64 values. */
typedef struct {
    double v;
    int32_t id;
} dentry_t;

static int dentry_order(const void* pa, const void* pb) {
    const dentry_t* a = (const dentry_t*)pa;
    const dentry_t* b = (const dentry_t*)pb;
    if (a->v != b->v) return a->v > b->v ? -1 : 1;
    return (a->id < b->id) ? -1 : (a->id > b->id ? 1 : 0);
}

static void lmhead_row(void* vctx, int64_t r) {
    lmhead_ctx* c = (lmhead_ctx*)vctx;
    dentry_t* e = (dentry_t*)malloc((size_t)c->V * sizeof(dentry_t));
    if (!e) {
        c->failed = 1;
        return;
    }
    const uint16_t* x = c->hidden + r * c->H;
    for (int64_t v = 0; v < c->V; ++v) {
        const uint16_t* w = c->lm_head + v * c->H;   /* LM head row v: [V, H] */
        double s = 0.0;
        for (int64_t i = 0; i < c->H; ++i) s += bf16_to_double(w[i]) * bf16_to_double(x[i]);
        e[v].v = s;
        e[v].id = (int32_t)v;
        if (c->logits_out) c->logits_out[r * c->V + v] = s;
    }
    qsort(e, (size_t)c->V, sizeof(dentry_t), dentry_order);
    for (int k = 0; k < c->K; ++k) {
        c->ids[r * c->K + k] = e[k].id;
        c->unary[r * c->K + k] = processed_logit((float)e[k].v, c->softcap, c->scale);
    }
    free(e);
}

/* The candidate head of DFlash2BeamForCausalLM.compute_candidates in full:
 * logits[r, v] = sum_i hidden[r, i] * lm_head[v, i] (exact, fp64), then the K first tokens
 * of the candidate order (logit descending, id ascending) and their processed logits.
 * logits_out (may be NULL) receives the exact logits [rows, V]. */
int oracle_lmhead_topk(const uint16_t* hidden, const uint16_t* lm_head, int64_t rows, int64_t H,
                       int64_t V, int K, double softcap, double scale, int32_t* ids, float* unary,
                       double* logits_out, int threads) {
    if (!hidden || !lm_head || !ids || !unary || rows < 0 || H < 1 || V < 1 || K < 1 || K > V)
        return -1;
    if (!(scale > 0.0)) return -1;
    lmhead_ctx c = {hidden, lm_head, H, V, K, softcap, scale, ids, unary, logits_out, 0};
    parallel_rows(lmhead_row, &c, rows, threads);
    return c.failed ? -1 : 0;
}

/* ---------------------------------------------------------------- step 2: projection */

typedef struct {
    const uint16_t* hidden;
    const uint16_t* w;
    int64_t H, rank;
    uint16_t* h_out;
    double* h_exact;
} proj_ctx;

static void proj_row(void* vctx, int64_t r) {
    proj_ctx* c = (proj_ctx*)vctx;
    const uint16_t* x = c->hidden + r * c->H;
    for (int64_t j = 0; j < c->rank; ++j) {
        const uint16_t* wj = c->w + j * c->H;      /* Linear weight [out = rank, in = H] */
        double s = 0.0;
        for (int64_t i = 0; i < c->H; ++i) s += bf16_to_double(wj[i]) * bf16_to_double(x[i]);
        c->h_out[r * c->rank + j] = oracle_bf16_round(s);
        if (c->h_exact) c->h_exact[r * c->rank + j] = s;
    }
}

/* h[r, j] = bf16( sum_i W[j, i] * hidden[r, i] ), with no bias.
 * hidden is [rows, H] and W is [rank, H], both as bf16 bit patterns; h_out is
 * [rows, rank] bf16. h_exact (may be NULL) receives the unrounded fp64 sums. */
int oracle_projection(const uint16_t* hidden, const uint16_t* w, int64_t rows, int64_t H,
                      int64_t rank, uint16_t* h_out, double* h_exact, int threads) {
    if (!hidden || !w || !h_out || rows < 0 || H < 1 || rank < 1) return -1;
    proj_ctx c = {hidden, w, H, rank, h_out, h_exact};
    parallel_rows(proj_row, &c, rows, threads);
    return 0;
}

/* ---------------------------------------------------------------- step 3: edge scores */

typedef struct {
    const uint16_t* pred_cb;
    const uint16_t* succ_cb;
    int64_t V, rank;
    const int32_t* cand;
    const float* unary;
    const uint16_t* h;
    const int32_t* anchors;
    int64_t S;
    int K;
    float* edges;
    int bad_id;
} edge_ctx;

static void edge_row(void* vctx, int64_t row) {
    edge_ctx* c = (edge_ctx*)vctx;
    const int64_t r = row / c->S, p = row % c->S;
    const int K = c->K;
    const uint16_t* hp = c->h + row * c->rank;
    for (int q = 0; q < K; ++q) {
        /* The predecessor of position p is candidate q of position p-1. At p = 0 it is
         * the anchor token, the same for every q. */
        const int64_t pid = (p == 0) ? c->anchors[r] : c->cand[(row - 1) * K + q];
        for (int cc = 0; cc < K; ++cc) {
            const int64_t cid = c->cand[row * K + cc];
            float* out = &c->edges[(row * K + q) * K + cc];
            if (pid < 0 || pid >= c->V || cid < 0 || cid >= c->V) {
                c->bad_id = 1;
                *out = NAN;
                continue;
            }
            const uint16_t* a = c->pred_cb + pid * c->rank;
            const uint16_t* b = c->succ_cb + cid * c->rank;
            double s = (double)c->unary[row * K + cc];
            for (int64_t j = 0; j < c->rank; ++j)
                s += bf16_to_double(a[j]) * bf16_to_double(hp[j]) * bf16_to_double(b[j]);
            *out = (float)s;
        }
    }
}

/* E[r, p, q, c] = unary[r, p, c] + sum_j pred_cb[pid, j] * h[r, p, j] * succ_cb[cid, j]
 * with cid = cand[r, p, c] and pid = cand[r, p-1, q] (p > 0) or anchors[r] (p = 0).
 * Codebooks are [V, rank] bf16 bits, cand/unary [R, S, K], h [R, S, rank] bf16 bits,
 * anchors [R], edges [R, S, K, K] fp32. Returns 0, 1 if an id was out of [0, V)
 * (those scores are NaN), or -1 on bad arguments. */
int oracle_edges(const uint16_t* pred_cb, const uint16_t* succ_cb, int64_t V, int64_t rank,
                 const int32_t* cand, const float* unary, const uint16_t* h,
                 const int32_t* anchors, int64_t R, int64_t S, int K, float* edges,
                 int threads) {
    if (!pred_cb || !succ_cb || !cand || !unary || !h || !anchors || !edges) return -1;
    if (V < 1 || rank < 1 || R < 0 || S < 1 || K < 1) return -1;
    edge_ctx c = {pred_cb, succ_cb, V, rank, cand, unary, h, anchors, S, K, edges, 0};
    parallel_rows(edge_row, &c, R * S, threads);
    return c.bad_id ? 1 : 0;
}

/* ---------------------------------------------------------------- all three steps */

/* The whole selector for R requests: top-k (with the processed unary), projection, edges.
 * Outputs as above; the edge scores use the processed unary values. */
int oracle_selector(const float* logits, const uint16_t* hidden, const uint16_t* w,
                    const uint16_t* pred_cb, const uint16_t* succ_cb, const int32_t* anchors,
                    int64_t R, int64_t S, int K, int64_t V, int64_t H, int64_t rank,
                    double softcap, double scale, int32_t* ids, float* unary, uint16_t* h_out,
                    float* edges, int threads) {
    int rc = oracle_topk(logits, R * S, V, K, softcap, scale, ids, unary, threads);
    if (rc) return rc;
    rc = oracle_projection(hidden, w, R * S, H, rank, h_out, NULL, threads);
    if (rc) return rc;
    return oracle_edges(pred_cb, succ_cb, V, rank, ids, unary, h_out, anchors, R, S, K, edges,
                        threads);
}

/* ---------------------------------------------------------------------------------
 * Best path over the edge scores. The pages say the selector rescores each step's top-k
 * candidates against the token before it; what consumes the scores is not shown. The
 * reading: for request r, choose one candidate index c_p per step p so that the sum over
 * p of E[r,p,c_{p-1},c_p] is largest, the predecessor row at p = 0 being q = 0 (every q row
 * is the anchor's there). Max-sum dynamic programming over the steps, in fp32, in this
 * order:
 *   V_0[c] = E[r,0,0,c];
 *   V_p[c] = the largest of V_{p-1}[q] + E[r,p,q,c] over q = 0, 1, ..., K-1, taken as a
 *            running maximum that a later q replaces only with a strictly larger sum (ties
 *            keep the lower q; IEEE compares, so a NaN neither replaces nor is replaced);
 *   c_{S-1} = the running maximum of V_{S-1}[c] over c, same rule; c_{p-1} = the q kept
 *            for (p, c_p).
 * Outputs: path[r,p] = c_p, tokens[r,p] = cand[r,p,c_p], score[r] = V_{S-1}[c_{S-1}].
 * The arithmetic is fp32 on purpose: a GPU that takes the same decisions in the same
 * precision and order gives the same path, bit for bit.
 * --------------------------------------------------------------------------------- */
typedef struct {
    const float* edges;
    const int32_t* cand;
    int64_t S;
    int K;
    int32_t* path;
    int32_t* tokens;
    float* score;
    int failed;
} PathCtx;

static void path_row(void* ctx, int64_t r) {
    PathCtx* c = (PathCtx*)ctx;
    const int K = c->K;
    const int64_t S = c->S;
    const float* E = c->edges + r * S * K * K;
    float v[32] = {0}, nv[32];
    unsigned char* keep = (unsigned char*)malloc((size_t)(S * K));
    if (!keep) {
        c->failed = 1;
        return;
    }
    for (int j = 0; j < K; ++j) v[j] = E[j];                 /* p = 0, predecessor row q = 0 */
    for (int64_t p = 1; p < S; ++p) {
        const float* Ep = E + p * K * K;
        for (int j = 0; j < K; ++j) {
            float best = v[0] + Ep[j];
            int bq = 0;
            for (int q = 1; q < K; ++q) {
                const float s = v[q] + Ep[q * K + j];
                if (s > best) {
                    best = s;
                    bq = q;
                }
            }
            nv[j] = best;
            keep[p * K + j] = (unsigned char)bq;
        }
        memcpy(v, nv, sizeof(float) * (size_t)K);
    }
    int cur = 0;
    for (int j = 1; j < K; ++j)
        if (v[j] > v[cur]) cur = j;
    c->score[r] = v[cur];
    for (int64_t p = S - 1; p >= 0; --p) {
        c->path[r * S + p] = cur;
        c->tokens[r * S + p] = c->cand[(r * S + p) * K + cur];
        if (p > 0) cur = keep[p * K + cur];
    }
    free(keep);
}

int oracle_best_path(const float* edges, const int32_t* cand, int64_t R, int64_t S, int K,
                     int32_t* path, int32_t* tokens, float* score, int threads) {
    if (R < 1 || S < 1 || K < 1 || K > 32) return -1;
    PathCtx c = {edges, cand, S, K, path, tokens, score, 0};
    parallel_rows(path_row, &c, R, threads);
    return c.failed ? -2 : 0;
}
