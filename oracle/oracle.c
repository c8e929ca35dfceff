/*
 * oracle.c -- plain, slow, obviously correct CPU reference of the
 * lightning-indexer hot path.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Every function is the plain definition written out in fp64 loops; the only
 * library primitives are qsort (top-k ordering) and rint (nearest-even).
 * Parallelism is over independent rows only; there is no blocking, fusion or
 * reordering of any sum beyond the per-row loops written here.
 *
 * Sources (indexer documentation pages):
 *   "tilelang_indexer" page, V4IndexerFunction / v4_lighting_indexer: layouts,
 *     compress_ratio, topk, optional topk_indices, backward(grad_scores, ...).
 *   "tilelang_indexer" page, pytorch_extract_topk_scores: gather at indices.
 *   "tilelang_indexer_fwd" page, _make_causal_cu_seqlens: query p sees
 *     compressed groups [0, (p+1)//compress_ratio).
 *   "tilelang_indexer_fwd" page, batched_indexer_fwd / indexer_fwd_interface /
 *     clean_logits_: [seqlen, seqlen_kv] fp32 logits over [ks, ke).
 *   "deepseek_v41.indexer" page, module docstring and indexer_scores: bf16
 *     rounding of the GEMM result and of the weighted head score, fp32 reduce,
 *     boolean visibility, bf16 scores.
 */
#define _DEFAULT_SOURCE 1
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------ threads */
static int g_threads = 0;

void orc_set_threads(int n) { g_threads = n; }

int orc_get_threads(void) {
    if (g_threads > 0) return g_threads;
    long n = 1;
#ifdef _SC_NPROCESSORS_ONLN
    n = sysconf(_SC_NPROCESSORS_ONLN);
#endif
    return n > 0 ? (int)n : 1;
}

typedef void (*row_fn)(void* ctx, int64_t i, int tid);

typedef struct {
    row_fn fn;
    void* ctx;
    int64_t n;
    int tid;
    int nthreads;
} worker_arg;

static void* worker_main(void* p) {
    worker_arg* a = (worker_arg*)p;
    for (int64_t i = a->tid; i < a->n; i += a->nthreads) a->fn(a->ctx, i, a->tid);
    return NULL;
}

/* Runs fn(ctx, i, tid) for i in [0, n) over the oracle's threads. */
static void parallel_rows(int64_t n, row_fn fn, void* ctx, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    pthread_t th[512];
    worker_arg args[512];
    if (nthreads > 512) nthreads = 512;
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn; args[t].ctx = ctx; args[t].n = n;
        args[t].tid = t; args[t].nthreads = nthreads;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, worker_main, &args[t]);
    worker_main(&args[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* --------------------------------------------------------------------- bf16 */
/* A bf16 pattern is the upper 16 bits of an IEEE binary32 pattern. */
double orc_bf16_decode(uint16_t v) {
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round v to the nearest bf16 value (8 significant bits, exponent range of
 * binary32), ties to even, written from the IEEE 754 definition:
 * scale so the retained bits form the integer part, rint (ties-to-even in the
 * default rounding mode), scale back.  Below 2^-126 the quantum is fixed at
 * 2^-133 (subnormals).  Results beyond the largest finite bf16 become inf. */
double orc_bf16_round(double v) {
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    int e;
    frexp(v, &e);            /* v = m * 2^e, 0.5 <= |m| < 1 */
    int q = e - 8;           /* quantum exponent: 8 significant bits */
    if (q < -133) q = -133;  /* subnormal bf16 quantum */
    double r = ldexp(rint(ldexp(v, -q)), q);
    const double max_bf16 = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > max_bf16) return v > 0 ? INFINITY : -INFINITY;
    return r;
}

void orc_bf16_round_array(const double* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(in[i]);
}

static double act_f(double x, int act) { return act == ORC_ACT_RELU ? (x > 0.0 ? x : 0.0) : x; }
/* derivative; ReLU'(0) = 0 */
static double act_d(double x, int act) { return act == ORC_ACT_RELU ? (x > 0.0 ? 1.0 : 0.0) : 1.0; }

/* ------------------------------------------------------------ causal ranges */
void orc_causal_ranges(int64_t S, int64_t Skv, int ratio, int32_t* ks, int32_t* ke) {
    for (int64_t s = 0; s < S; ++s) {
        int64_t e = (s + 1) / ratio;
        if (e > Skv) e = Skv;
        ks[s] = 0;
        ke[s] = (int32_t)e;
    }
}

static void clamp_range(int32_t a, int32_t b, int64_t Skv, int64_t* lo, int64_t* hi) {
    int64_t l = a < 0 ? 0 : a, h = b > Skv ? Skv : b;
    if (h < l) h = l;
    *lo = l; *hi = h;
}

/* ------------------------------------------------------------------- logits */
typedef struct {
    const uint16_t *q, *k;
    const float* w;
    int64_t B, S, Skv;
    int H, D, act;
    const int32_t *ks, *ke;
    const int64_t* rows;
    double* out;
} logits_ctx;

static void logits_row(void* p, int64_t i, int tid) {
    (void)tid;
    logits_ctx* c = (logits_ctx*)p;
    int64_t r = c->rows[i], b = r / c->S, s = r % c->S;
    int64_t lo, hi;
    clamp_range(c->ks[s], c->ke[s], c->Skv, &lo, &hi);
    double* o = c->out + i * c->Skv;
    /* decoded copies of this row's queries and of one key row */
    double* qd = (double*)malloc(sizeof(double) * (size_t)c->H * (size_t)c->D);
    double* kd = (double*)malloc(sizeof(double) * (size_t)c->D);
    for (int h = 0; h < c->H; ++h)
        for (int d = 0; d < c->D; ++d)
            qd[h * c->D + d] = orc_bf16_decode(c->q[((s * c->B + b) * c->H + h) * c->D + d]);
    for (int64_t t = 0; t < c->Skv; ++t) o[t] = -INFINITY;
    for (int64_t t = lo; t < hi; ++t) {
        for (int d = 0; d < c->D; ++d) kd[d] = orc_bf16_decode(c->k[(t * c->B + b) * c->D + d]);
        double acc = 0.0;
        for (int h = 0; h < c->H; ++h) {
            double x = 0.0;
            for (int d = 0; d < c->D; ++d) x += qd[h * c->D + d] * kd[d];
            acc += (double)c->w[(s * c->B + b) * c->H + h] * act_f(x, c->act);
        }
        o[t] = acc;
    }
    free(qd);
    free(kd);
}

int orc_logits_rows(const uint16_t* q, const uint16_t* k, const float* w,
                    int64_t B, int64_t S, int64_t Skv, int H, int D,
                    const int32_t* ks, const int32_t* ke, int act,
                    const int64_t* rows, int64_t nrows, double* out) {
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= B * S) return 1;
    logits_ctx c = {q, k, w, B, S, Skv, H, D, act, ks, ke, rows, out};
    parallel_rows(nrows, logits_row, &c, orc_get_threads());
    return 0;
}

/* -------------------------------------------------------------------- top-k */
typedef struct {
    double v;
    int32_t t;
} cand;

/* score descending, then index ascending */
static int cand_cmp(const void* a, const void* b) {
    const cand* x = (const cand*)a;
    const cand* y = (const cand*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->t > y->t) - (x->t < y->t);
}

typedef struct {
    const double* logits;
    int64_t Skv, S;
    const int64_t* rows;
    const int32_t *ks, *ke;
    int topk;
    int32_t* idx;
    double* score;
    cand** scratch;
} topk_ctx;

static void topk_row(void* p, int64_t i, int tid) {
    topk_ctx* c = (topk_ctx*)p;
    int64_t s = c->rows[i] % c->S;
    int64_t lo, hi;
    clamp_range(c->ks[s], c->ke[s], c->Skv, &lo, &hi);
    cand* buf = c->scratch[tid];
    int64_t n = 0;
    for (int64_t t = lo; t < hi; ++t) {
        buf[n].v = c->logits[i * c->Skv + t];
        buf[n].t = (int32_t)t;
        ++n;
    }
    qsort(buf, (size_t)n, sizeof(cand), cand_cmp);
    for (int j = 0; j < c->topk; ++j) {
        if (j < n) {
            c->idx[i * c->topk + j] = buf[j].t;
            c->score[i * c->topk + j] = buf[j].v;
        } else {
            c->idx[i * c->topk + j] = -1;
            c->score[i * c->topk + j] = -INFINITY;
        }
    }
}

int orc_topk_rows(const double* logits, int64_t nrows, int64_t Skv,
                  const int64_t* rows, int64_t S, const int32_t* ks, const int32_t* ke,
                  int topk, int32_t* idx_out, double* score_out) {
    if (topk < 0) return 1;
    int nt = orc_get_threads();
    if (nt > 512) nt = 512;
    cand* scratch[512];
    for (int t = 0; t < nt; ++t) {
        scratch[t] = (cand*)malloc(sizeof(cand) * (size_t)(Skv > 0 ? Skv : 1));
        if (!scratch[t]) {
            for (int u = 0; u < t; ++u) free(scratch[u]);
            return 2;
        }
    }
    topk_ctx c = {logits, Skv, S, rows, ks, ke, topk, idx_out, score_out, scratch};
    parallel_rows(nrows, topk_row, &c, nt);
    for (int t = 0; t < nt; ++t) free(scratch[t]);
    return 0;
}

/* Top-k over the entries of each row whose mask byte is nonzero ("deepseek_v41.
 * indexer" page, module docstring: the top-k / candidate selection runs on the
 * scorer's output over the visible keys).  Same order and padding as
 * orc_topk_rows. */
typedef struct {
    const double* logits;
    const uint8_t* mask;
    int64_t Skv;
    int topk;
    int32_t* idx;
    double* score;
    cand** scratch;
} topk_masked_ctx;

static void topk_masked_row(void* p, int64_t i, int tid) {
    topk_masked_ctx* c = (topk_masked_ctx*)p;
    cand* buf = c->scratch[tid];
    int64_t n = 0;
    for (int64_t t = 0; t < c->Skv; ++t) {
        if (!c->mask[i * c->Skv + t]) continue;
        buf[n].v = c->logits[i * c->Skv + t];
        buf[n].t = (int32_t)t;
        ++n;
    }
    qsort(buf, (size_t)n, sizeof(cand), cand_cmp);
    for (int j = 0; j < c->topk; ++j) {
        if (j < n) {
            c->idx[i * c->topk + j] = buf[j].t;
            c->score[i * c->topk + j] = buf[j].v;
        } else {
            c->idx[i * c->topk + j] = -1;
            c->score[i * c->topk + j] = -INFINITY;
        }
    }
}

int orc_topk_masked_rows(const double* logits, const uint8_t* mask, int64_t nrows, int64_t Skv,
                         int topk, int32_t* idx_out, double* score_out) {
    if (topk < 0) return 1;
    int nt = orc_get_threads();
    if (nt > 512) nt = 512;
    cand* scratch[512];
    for (int t = 0; t < nt; ++t) {
        scratch[t] = (cand*)malloc(sizeof(cand) * (size_t)(Skv > 0 ? Skv : 1));
        if (!scratch[t]) {
            for (int u = 0; u < t; ++u) free(scratch[u]);
            return 2;
        }
    }
    topk_masked_ctx c = {logits, mask, Skv, topk, idx_out, score_out, scratch};
    parallel_rows(nrows, topk_masked_row, &c, nt);
    for (int t = 0; t < nt; ++t) free(scratch[t]);
    return 0;
}

/* ------------------------------------------------------------------ extract */
void orc_extract_rows(const double* logits, int64_t nrows, int64_t Skv,
                      const int32_t* idx, int topk, double* out) {
    for (int64_t i = 0; i < nrows; ++i)
        for (int j = 0; j < topk; ++j) {
            int32_t t = idx[i * topk + j];
            out[i * topk + j] = (t >= 0 && t < Skv) ? logits[i * Skv + t] : -INFINITY;
        }
}

/* ------------------------------------------------------- scores at indices */
typedef struct {
    const uint16_t *q, *k;
    const float* w;
    int64_t B, S, Skv;
    int H, D, act;
    const int32_t *ks, *ke;
    const int64_t* rows;
    const int32_t* idx;
    int topk;
    double* out;
} gather_ctx;

static void gather_row(void* p, int64_t i, int tid) {
    (void)tid;
    gather_ctx* c = (gather_ctx*)p;
    int64_t r = c->rows[i], b = r / c->S, s = r % c->S;
    int64_t lo, hi;
    clamp_range(c->ks[s], c->ke[s], c->Skv, &lo, &hi);
    for (int j = 0; j < c->topk; ++j) {
        int64_t t = c->idx[i * c->topk + j];
        if (t < lo || t >= hi) {
            c->out[i * c->topk + j] = -INFINITY;
            continue;
        }
        const uint16_t* kr = c->k + (t * c->B + b) * c->D;
        double acc = 0.0;
        for (int h = 0; h < c->H; ++h) {
            const uint16_t* qr = c->q + ((s * c->B + b) * c->H + h) * c->D;
            double x = 0.0;
            for (int d = 0; d < c->D; ++d) x += orc_bf16_decode(qr[d]) * orc_bf16_decode(kr[d]);
            acc += (double)c->w[(s * c->B + b) * c->H + h] * act_f(x, c->act);
        }
        c->out[i * c->topk + j] = acc;
    }
}

int orc_gather_scores_rows(const uint16_t* q, const uint16_t* k, const float* w,
                           int64_t B, int64_t S, int64_t Skv, int H, int D,
                           const int32_t* ks, const int32_t* ke, int act,
                           const int64_t* rows, int64_t nrows,
                           const int32_t* idx, int topk, double* out) {
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= B * S) return 1;
    gather_ctx c = {q, k, w, B, S, Skv, H, D, act, ks, ke, rows, idx, topk, out};
    parallel_rows(nrows, gather_row, &c, orc_get_threads());
    return 0;
}

/* -------------------------------------------------------------------- V4.1 */
typedef struct {
    const uint16_t *q, *k, *w;
    const uint8_t* allowed;
    int64_t B, S, Skv;
    int H, D, act;
    const int64_t* rows;
    float* out;
} v41_ctx;

static void v41_row(void* p, int64_t i, int tid) {
    (void)tid;
    v41_ctx* c = (v41_ctx*)p;
    int64_t r = c->rows[i], b = r / c->S, s = r % c->S;
    double* qd = (double*)malloc(sizeof(double) * (size_t)c->H * (size_t)c->D);
    double* kd = (double*)malloc(sizeof(double) * (size_t)c->D);
    for (int h = 0; h < c->H; ++h)
        for (int d = 0; d < c->D; ++d)
            qd[h * c->D + d] = orc_bf16_decode(c->q[((b * c->S + s) * c->H + h) * c->D + d]);
    const uint8_t* vis = c->allowed + (b * c->S + s) * c->Skv;
    float* o = c->out + i * c->Skv;
    for (int64_t t = 0; t < c->Skv; ++t) {
        if (!vis[t]) {
            o[t] = -INFINITY;
            continue;
        }
        for (int d = 0; d < c->D; ++d) kd[d] = orc_bf16_decode(c->k[(b * c->Skv + t) * c->D + d]);
        double sum = 0.0;
        for (int h = 0; h < c->H; ++h) {
            double x = 0.0;
            for (int d = 0; d < c->D; ++d) x += qd[h * c->D + d] * kd[d];
            double y = orc_bf16_round(x);                        /* GEMM result -> bf16 */
            double wv = orc_bf16_decode(c->w[(b * c->S + s) * c->H + h]);
            double z = orc_bf16_round(act_f(y, c->act) * wv);    /* weighted head score -> bf16 */
            sum += z;                                            /* head reduction */
        }
        o[t] = (float)orc_bf16_round(sum);                       /* bf16 score */
    }
    free(qd);
    free(kd);
}

int orc_scores_v41_rows(const uint16_t* q, const uint16_t* k, const uint16_t* w,
                        const uint8_t* allowed, int64_t B, int64_t S, int64_t Skv,
                        int H, int D, int act, const int64_t* rows, int64_t nrows,
                        float* out) {
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= B * S) return 1;
    v41_ctx c = {q, k, w, allowed, B, S, Skv, H, D, act, rows, out};
    parallel_rows(nrows, v41_row, &c, orc_get_threads());
    return 0;
}

/* ---------------------------------------------------------------- backward */
typedef struct {
    const uint16_t *q, *k;
    const float *w, *grad;
    const int32_t* idx;
    int64_t B, S, Skv;
    int H, D, topk, act;
    const int32_t *ks, *ke;
    double gamma;
    double *dq, *dw, *dq_slack, *dw_slack;
    double **dk_part, **dk_slack_part; /* per thread [Skv*B*D] */
} bwd_ctx;

static void bwd_row(void* p, int64_t r, int tid) {
    bwd_ctx* c = (bwd_ctx*)p;
    int64_t b = r / c->S, s = r % c->S;
    int64_t lo, hi;
    clamp_range(c->ks[s], c->ke[s], c->Skv, &lo, &hi);
    const int H = c->H, D = c->D;
    double* dk = c->dk_part[tid];
    double* dks = c->dk_slack_part ? c->dk_slack_part[tid] : NULL;
    for (int j = 0; j < c->topk; ++j) {
        int64_t t = c->idx[r * c->topk + j];
        if (t < lo || t >= hi) continue; /* padding or invisible: no gradient */
        double g = (double)c->grad[r * c->topk + j];
        for (int h = 0; h < H; ++h) {
            int64_t qo = ((s * c->B + b) * H + h) * D, ko = (t * c->B + b) * D;
            double x = 0.0, mag = 0.0;
            for (int d = 0; d < D; ++d) {
                double pr = orc_bf16_decode(c->q[qo + d]) * orc_bf16_decode(c->k[ko + d]);
                x += pr;
                mag += fabs(pr);
            }
            int64_t wo = (s * c->B + b) * H + h;
            double wv = (double)c->w[wo];
            int ambiguous = c->act == ORC_ACT_RELU && fabs(x) <= c->gamma * mag;
            double a = act_f(x, c->act);
            c->dw[wo] += g * a;
            if (ambiguous && c->dw_slack) c->dw_slack[wo] += fabs(g) * c->gamma * mag;
            double cc = g * wv * act_d(x, c->act);
            /* for an ambiguous pair the other ReLU branch would add g*w */
            double amb = ambiguous ? fabs(g * wv) : 0.0;
            for (int d = 0; d < D; ++d) {
                double kv = orc_bf16_decode(c->k[ko + d]), qv = orc_bf16_decode(c->q[qo + d]);
                c->dq[qo + d] += cc * kv;
                dk[ko + d] += cc * qv;
                if (amb > 0.0) {
                    if (c->dq_slack) c->dq_slack[qo + d] += amb * fabs(kv);
                    if (dks) dks[ko + d] += amb * fabs(qv);
                }
            }
        }
    }
}

int orc_bwd(const uint16_t* q, const uint16_t* k, const float* w,
            const int32_t* idx, const float* grad,
            int64_t B, int64_t S, int64_t Skv, int H, int D,
            const int32_t* ks, const int32_t* ke, int topk, int act, double gamma,
            double* dq, double* dk, double* dw,
            double* dq_slack, double* dk_slack, double* dw_slack) {
    int64_t nq = S * B * H * D, nk = Skv * B * D, nw = S * B * H;
    memset(dq, 0, sizeof(double) * (size_t)nq);
    memset(dk, 0, sizeof(double) * (size_t)nk);
    memset(dw, 0, sizeof(double) * (size_t)nw);
    if (dq_slack) memset(dq_slack, 0, sizeof(double) * (size_t)nq);
    if (dk_slack) memset(dk_slack, 0, sizeof(double) * (size_t)nk);
    if (dw_slack) memset(dw_slack, 0, sizeof(double) * (size_t)nw);
    int nt = orc_get_threads();
    if (nt > 64) nt = 64;
    double* part[64];
    double* spart[64];
    for (int t = 0; t < nt; ++t) {
        part[t] = (double*)calloc((size_t)(nk > 0 ? nk : 1), sizeof(double));
        spart[t] = dk_slack ? (double*)calloc((size_t)(nk > 0 ? nk : 1), sizeof(double)) : NULL;
        if (!part[t] || (dk_slack && !spart[t])) return 2;
    }
    bwd_ctx c = {q, k, w, grad, idx, B, S, Skv, H, D, topk, act, ks, ke, gamma,
                 dq, dw, dq_slack, dw_slack, part, dk_slack ? spart : NULL};
    /* rows are independent for dq and dw; dk sums per-thread partials */
    parallel_rows(B * S, bwd_row, &c, nt);
    for (int t = 0; t < nt; ++t) {
        for (int64_t i = 0; i < nk; ++i) dk[i] += part[t][i];
        if (dk_slack)
            for (int64_t i = 0; i < nk; ++i) dk_slack[i] += spart[t][i];
        free(part[t]);
        free(spart[t]);
    }
    return 0;
}
