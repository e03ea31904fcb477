/*
 * CPU oracle for per-row vocabulary selection.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously-correct statement of what the GPU
 * library computes.  It shares no code, header, table or constant generator
 * with the CUDA path.  Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline / reference arm may load it; the product path never
 * does.
 *
 * Everything is computed in double, every row is fully sorted, and cumulative
 * masses are explicit running sums over that sorted order.
 *
 * Sources (page title, section):
 *   logits-processor, "API" and "Method": bitmask apply (bit 1 = allowed), the
 *     top-k / top-p / min-p keep sets resolved as one keep-threshold, the
 *     intersection of the three filters, greedy for temperature <= 0, the
 *     Gumbel-max draw keyed by (seed, row, offset).
 *   logits-mask-xpu, "Method" and "Validation": top_k == 1 dispatched to argmax,
 *     top_p = 1 keeps the full support.
 *   lm-head-topk, "API", "Method" and "Correctness": exact top-k sorted
 *     descending, ties to the lower vocabulary index, k <= 2048.
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *     Easy as 1, 2, 3", SC'11 (the Philox construction, N = 4, W = 32, R = 10).
 *
 * Readings where the pages are silent (the library makes the same ones):
 *   - counter layout: key = (seed lo, seed hi), counter = (i >> 2, row,
 *     offset lo, offset hi); token i takes output word i & 3;
 *   - uniform u = (2 * (x >> 9) + 1) * 2^-24, on the odd lattice of
 *     [2^-24, 1 - 2^-24]; E = -ln u (as -log1p(-(1-u)) for u >= 1/2);
 *     Gumbel G = -ln E;
 *   - keep sets keep whole tie groups at their boundary; the argmax class is
 *     always kept by top-p and min-p; top-k ranks raw logits;
 *   - a row with no allowed finite logit yields token -1;
 *   - bit order inside a mask word is LSB-first (token i is bit i & 31 of
 *     word i >> 5); bits at or beyond V are ignored.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TSAO_OK 0
#define TSAO_ERR_NAN (-1)
#define TSAO_ERR_ARG (-2)
#define TSAO_ERR_NOMEM (-3)

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11).  One round maps the counter
 * (c0, c1, c2, c3) with key (k0, k1) to
 *   (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0)),
 * and the key is bumped by the Weyl increments (W0, W1) between rounds.      */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u /* golden ratio */
#define PHILOX_W1 0xBB67AE85u /* sqrt(3) - 1 */

void tsao_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32-bit random word of token i in row b for draw (seed, offset). */
uint32_t tsao_rand_word(uint64_t seed, uint64_t offset, int64_t b, int64_t i) {
    uint32_t ctr[4] = {(uint32_t)((uint64_t)i >> 2), (uint32_t)b, (uint32_t)offset,
                       (uint32_t)(offset >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    tsao_philox4x32_10(ctr, key, out);
    return out[i & 3];
}

/* Words of tokens i0 .. i0 + n - 1 of row b (a batch of tsao_rand_word). */
void tsao_rand_words(uint64_t seed, uint64_t offset, int64_t b, int64_t i0, int64_t n,
                     uint32_t *out) {
    for (int64_t t = 0; t < n; ++t) out[t] = tsao_rand_word(seed, offset, b, i0 + t);
}

/* u on the odd lattice: never 0, never 1. */
double tsao_uniform(uint32_t x) { return (2.0 * (double)(x >> 9) + 1.0) * 0x1p-24; }

/* Standard Gumbel variate G = -ln(-ln u). */
double tsao_gumbel(uint32_t x) {
    double u = tsao_uniform(x);
    double e = (u < 0.5) ? -log(u) : -log1p(-(1.0 - u));
    return -log(e);
}

/* ------------------------------------------------------------------------ */
/* logits-processor, "API": apply_token_bitmask sets the disallowed logits to
 * -inf in place; bit 1 = allowed.  dtype 0 = f32, 1 = f16, 2 = bf16.          */
int tsao_apply_token_bitmask(void *logits, int dtype, int64_t B, int64_t V, int64_t stride,
                             const int32_t *mask, int64_t mstride) {
    if (B < 0 || V < 0 || stride < V || mstride < (V + 31) / 32) return TSAO_ERR_ARG;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t i = 0; i < V; ++i) {
            uint32_t word = (uint32_t)mask[b * mstride + (i >> 5)];
            int allowed = (word >> (i & 31)) & 1u;
            if (allowed) continue;
            if (dtype == 0) {
                uint32_t ninf = 0xFF800000u;
                memcpy((char *)logits + 4 * (b * stride + i), &ninf, 4);
            } else if (dtype == 1) {
                uint16_t ninf = 0xFC00u;
                memcpy((char *)logits + 2 * (b * stride + i), &ninf, 2);
            } else if (dtype == 2) {
                uint16_t ninf = 0xFF80u;
                memcpy((char *)logits + 2 * (b * stride + i), &ninf, 2);
            } else {
                return TSAO_ERR_ARG;
            }
        }
    }
    return TSAO_OK;
}

/* ------------------------------------------------------------------------ */
typedef struct {
    double l;
    int64_t i;
} entry;

/* Order by logit descending, then vocabulary index ascending.  -0.0 and +0.0
 * compare equal and fall back to the index. */
static int cmp_desc(const void *pa, const void *pb) {
    const entry *a = (const entry *)pa, *b = (const entry *)pb;
    if (a->l > b->l) return -1;
    if (a->l < b->l) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i);
}

typedef struct {
    int64_t token;   /* -1 when no allowed finite logit */
    double vstar;    /* smallest kept logit (NaN for an empty row) */
    double gap;      /* best minus second-best perturbed score over the keep set */
    double m, Z;     /* max logit, sum of exp((l - m) / T) over the allowed set */
    double v_k, v_p, v_m; /* per-filter thresholds; -inf when a filter keeps all */
    int64_t n_allowed, n_kept;
} row_result;

/* One row of `sample`, written out step by step (logits-processor, "Method";
 * the readings above).  M_out / w_out, when given, receive per token the mass
 * strictly above it (as a probability) and exp((l - m) / T); NaN / 0 for tokens
 * outside the allowed set. */
static int sample_row(const double *row, int64_t V, const int32_t *mrow, double T, int32_t top_k,
                      double top_p, double min_p, int sequential, uint64_t seed, uint64_t offset,
                      int64_t b, entry *ent, row_result *res, double *M_out, double *w_out) {
    /* 1. The allowed set A: mask bit 1 and a finite logit. */
    int64_t n = 0;
    for (int64_t i = 0; i < V; ++i) {
        double l = row[i];
        if (isnan(l)) return TSAO_ERR_NAN;
        if (M_out) M_out[i] = NAN;
        if (w_out) w_out[i] = 0.0;
        int allowed = mrow ? (int)(((uint32_t)mrow[i >> 5] >> (i & 31)) & 1u) : 1;
        if (!allowed || isinf(l)) continue;
        ent[n].l = l;
        ent[n].i = i;
        ++n;
    }
    res->n_allowed = n;
    res->gap = NAN;
    res->v_k = res->v_p = res->v_m = -INFINITY;
    res->Z = NAN;
    if (n == 0) {
        res->token = -1;
        res->vstar = NAN;
        res->m = -INFINITY;
        res->n_kept = 0;
        return TSAO_OK;
    }
    /* 2. Full sort by (logit desc, index asc). */
    qsort(ent, (size_t)n, sizeof(entry), cmp_desc);
    double m = ent[0].l;
    res->m = m;

    /* 3. Greedy: temperature <= 0, or top_k == 1 dispatched to argmax. */
    if (T <= 0.0 || top_k == 1) {
        res->token = ent[0].i;
        res->vstar = m;
        res->n_kept = 1;
        return TSAO_OK;
    }

    /* 4. Softmax weights w = exp(s - s_max) with s = l / T, and Z = sum w. */
    double Z = 0.0;
    for (int64_t j = 0; j < n; ++j) Z += exp((ent[j].l - m) / T);
    res->Z = Z;

    /* 5. Keep thresholds.  top-k: the k-th largest logit with multiplicity. */
    double v_k = -INFINITY;
    if (top_k >= 1 && (int64_t)top_k < n) v_k = ent[top_k - 1].l;

    /* top-p and min-p walk the tie groups in descending order with an explicit
     * running sum of the mass strictly above the group.  Top-p measures that
     * mass against Z, or -- in the sequential reading (logits-processor: the
     * transformers processor chain, where top-p sees the renormalised top-k
     * survivors) -- against the survivors' total Zp when top-k is active. */
    double Zp = Z;
    if (sequential && v_k > -INFINITY) {
        Zp = 0.0;
        for (int64_t t = 0; t < n && ent[t].l >= v_k; ++t) Zp += exp((ent[t].l - m) / T);
    }
    double v_p = -INFINITY, v_m = -INFINITY;
    int p_on = top_p < 1.0, m_on = min_p > 0.0;
    int p_open = 1, m_open = 1;
    double above = 0.0; /* sum of w over groups strictly above the current one */
    int64_t j = 0;
    int first = 1;
    while (j < n) {
        int64_t j1 = j;
        while (j1 < n && ent[j1].l == ent[j].l) ++j1;
        double w = exp((ent[j].l - m) / T);
        double M = above / Zp;
        if (M_out || w_out) {
            for (int64_t t = j; t < j1; ++t) {
                if (M_out) M_out[ent[t].i] = M;
                if (w_out) w_out[ent[t].i] = w;
            }
        }
        if (p_on && p_open) {
            if (first || M < top_p) v_p = ent[j].l;
            else p_open = 0;
        }
        if (m_on && m_open) {
            if (first || w >= min_p) v_m = ent[j].l;
            else m_open = 0;
        }
        for (int64_t t = j; t < j1; ++t) above += exp((ent[t].l - m) / T);
        first = 0;
        j = j1;
    }
    res->v_k = v_k;
    res->v_p = v_p;
    res->v_m = v_m;

    /* 6. The intersection of upward-closed sets is one threshold. */
    double vs = v_k;
    if (v_p > vs) vs = v_p;
    if (v_m > vs) vs = v_m;
    int64_t nk = 0;
    while (nk < n && ent[nk].l >= vs) ++nk;
    res->n_kept = nk;
    res->vstar = ent[nk - 1].l;

    /* 7. Gumbel-max over the keep set; exact score ties go to the lower index. */
    double best = -INFINITY, second = -INFINITY;
    int64_t best_i = -1;
    for (int64_t t = 0; t < nk; ++t) {
        int64_t i = ent[t].i;
        double score = ent[t].l / T + tsao_gumbel(tsao_rand_word(seed, offset, b, i));
        if (best_i < 0 || score > best || (score == best && i < best_i)) {
            second = best;
            best = score;
            best_i = i;
        } else if (score > second) {
            second = score;
        }
    }
    res->token = best_i;
    res->gap = (nk > 1) ? best - second : INFINITY;
    return TSAO_OK;
}

/* ------------------------------------------------------------------------ */
/* Row-parallel driver: rows are split statically over plain pthreads.       */
typedef struct {
    const double *logits;
    int64_t B, V, stride;
    const int32_t *mask;
    int64_t mstride;
    const double *T;
    const int32_t *top_k;
    const double *top_p, *min_p;
    uint64_t seed, offset;
    int64_t *tokens;
    double *vstar, *gap;
    int sequential;
    int64_t b0, b1;
    int status;
} sample_job;

static void *sample_worker(void *arg) {
    sample_job *job = (sample_job *)arg;
    entry *ent = (entry *)malloc(sizeof(entry) * (size_t)(job->V > 0 ? job->V : 1));
    if (!ent) {
        job->status = TSAO_ERR_NOMEM;
        return NULL;
    }
    for (int64_t b = job->b0; b < job->b1; ++b) {
        row_result r;
        const int32_t *mrow = job->mask ? job->mask + b * job->mstride : NULL;
        int st = sample_row(job->logits + b * job->stride, job->V, mrow, job->T[b], job->top_k[b],
                            job->top_p[b], job->min_p[b], job->sequential, job->seed,
                            job->offset, b, ent, &r, NULL, NULL);
        if (st != TSAO_OK) {
            job->status = st;
            break;
        }
        job->tokens[b] = r.token;
        if (job->vstar) job->vstar[b] = r.vstar;
        if (job->gap) job->gap[b] = r.gap;
    }
    free(ent);
    return NULL;
}

/* logits-processor, "API": sample(logits, temperature, top_k, top_p, min_p,
 * seed, offset) with every sampling parameter given per row ([B] arrays).
 * vstar / gap may be NULL.  sequential != 0 takes top-p over the renormalised
 * top-k survivors (the transformers chain) instead of the full softmax. */
int tsao_sample(const double *logits, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                int64_t mstride, const double *T, const int32_t *top_k, const double *top_p,
                const double *min_p, uint64_t seed, uint64_t offset, int64_t *tokens,
                double *vstar, double *gap, int nthreads, int sequential) {
    if (B < 0 || V < 1 || stride < V || (mask && mstride < (V + 31) / 32)) return TSAO_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = (int)(B > 0 ? B : 1);
    sample_job *jobs = (sample_job *)calloc((size_t)nthreads, sizeof(sample_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return TSAO_ERR_NOMEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        sample_job *jb = &jobs[t];
        jb->logits = logits; jb->B = B; jb->V = V; jb->stride = stride;
        jb->mask = mask; jb->mstride = mstride;
        jb->T = T; jb->top_k = top_k; jb->top_p = top_p; jb->min_p = min_p;
        jb->seed = seed; jb->offset = offset;
        jb->tokens = tokens; jb->vstar = vstar; jb->gap = gap;
        jb->sequential = sequential;
        jb->b0 = B * t / nthreads;
        jb->b1 = B * (t + 1) / nthreads;
        jb->status = TSAO_OK;
    }
    int status = TSAO_OK;
    if (nthreads == 1) {
        sample_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&th[t], NULL, sample_worker, &jobs[t]) != 0) break;
            ++started;
        }
        for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
        for (int t = started; t < nthreads; ++t) sample_worker(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != TSAO_OK) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

/* Every intermediate of one row, for the tests' tolerance rules.  out7 =
 * {m, Z, v_k, v_p, v_m, vstar, gap}; counts2 = {n_allowed, n_kept}.          */
int tsao_sample_row_detail(const double *row, int64_t V, const int32_t *mrow, double T,
                           int32_t top_k, double top_p, double min_p, uint64_t seed,
                           uint64_t offset, int64_t b, int64_t *token, double *out7,
                           int64_t *counts2, double *M_out, double *w_out, int sequential) {
    if (V < 1) return TSAO_ERR_ARG;
    entry *ent = (entry *)malloc(sizeof(entry) * (size_t)V);
    if (!ent) return TSAO_ERR_NOMEM;
    row_result r;
    int st = sample_row(row, V, mrow, T, top_k, top_p, min_p, sequential, seed, offset, b, ent, &r,
                        M_out, w_out);
    free(ent);
    if (st != TSAO_OK) return st;
    *token = r.token;
    out7[0] = r.m; out7[1] = r.Z; out7[2] = r.v_k; out7[3] = r.v_p;
    out7[4] = r.v_m; out7[5] = r.vstar; out7[6] = r.gap;
    counts2[0] = r.n_allowed; counts2[1] = r.n_kept;
    return TSAO_OK;
}

/* ------------------------------------------------------------------------ */
/* lm-head-topk, "API" / "Method": the k largest entries of each row sorted by
 * (value desc, index asc) -- the first k of the fully sorted row.            */
typedef struct {
    const double *logits;
    int64_t V, stride;
    int32_t k;
    double *values;
    int64_t *indices;
    int64_t b0, b1;
    int status;
} topk_job;

static void *topk_worker(void *arg) {
    topk_job *job = (topk_job *)arg;
    entry *ent = (entry *)malloc(sizeof(entry) * (size_t)job->V);
    if (!ent) {
        job->status = TSAO_ERR_NOMEM;
        return NULL;
    }
    for (int64_t b = job->b0; b < job->b1; ++b) {
        const double *row = job->logits + b * job->stride;
        for (int64_t i = 0; i < job->V; ++i) {
            if (isnan(row[i])) {
                job->status = TSAO_ERR_NAN;
                free(ent);
                return NULL;
            }
            ent[i].l = row[i];
            ent[i].i = i;
        }
        qsort(ent, (size_t)job->V, sizeof(entry), cmp_desc);
        for (int32_t j = 0; j < job->k; ++j) {
            job->values[b * job->k + j] = ent[j].l;
            job->indices[b * job->k + j] = ent[j].i;
        }
    }
    free(ent);
    return NULL;
}

int tsao_topk(const double *logits, int64_t B, int64_t V, int64_t stride, int32_t k,
              double *values, int64_t *indices, int nthreads) {
    if (B < 0 || V < 1 || stride < V || k < 1 || (int64_t)k > V || k > 2048) return TSAO_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = (int)(B > 0 ? B : 1);
    topk_job *jobs = (topk_job *)calloc((size_t)nthreads, sizeof(topk_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return TSAO_ERR_NOMEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        topk_job *jb = &jobs[t];
        jb->logits = logits; jb->V = V; jb->stride = stride; jb->k = k;
        jb->values = values; jb->indices = indices;
        jb->b0 = B * t / nthreads;
        jb->b1 = B * (t + 1) / nthreads;
        jb->status = TSAO_OK;
    }
    if (nthreads == 1) {
        topk_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&th[t], NULL, topk_worker, &jobs[t]) != 0) break;
            ++started;
        }
        for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
        for (int t = started; t < nthreads; ++t) topk_worker(&jobs[t]);
    }
    int status = TSAO_OK;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != TSAO_OK) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

/* ------------------------------------------------------------------------ */
/* logits-mask-xpu, "Usage" (bitmask_from_allowed): a [B, V] bool allow-set
 * packed into [B, ceil(V/32)] int32 words; token i is bit (i mod 32) of word
 * floor(i / 32) (the XGrammar token-bitmask convention that apply_token_bitmask
 * reads); the bits of the last word past V are 0.  allowed holds one byte per
 * token, nonzero for allowed.                                                 */
int tsao_bitmask_from_allowed(const uint8_t *allowed, int64_t B, int64_t V, int64_t astride,
                              int32_t *bits, int64_t wstride) {
    int64_t W = (V + 31) / 32;
    if (B < 0 || V < 1 || astride < V || wstride < W) return TSAO_ERR_ARG;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t w = 0; w < W; ++w) {
            uint32_t word = 0;
            for (int j = 0; j < 32; ++j) {
                int64_t i = w * 32 + j;
                if (i < V && allowed[b * astride + i] != 0) word |= 1u << j;
            }
            bits[b * wstride + w] = (int32_t)word;
        }
    }
    return TSAO_OK;
}

/* logits-mask-xpu, "Method" (the inverse-CDF draw) and "Usage" (a caller
 * uniform per row).  The keep set is the one `sample` forms: every allowed
 * finite logit >= v*.  Its weights are w_i = exp((l_i - m) / T).  Walking the
 * kept tokens in index order with the running sum S_i of their weights, the
 * token is the first one with S_i > u W, W the kept total (the last kept token
 * when no sum passes it).  Greedy rows (T <= 0, top_k == 1) and empty rows
 * give what `sample` gives.  Per row, vstar receives v* and W the kept total;
 * cum (when given, [B, V]) receives S_i at kept tokens and NaN elsewhere.    */
typedef struct {
    const double *logits;
    int64_t V, stride;
    const int32_t *mask;
    int64_t mstride;
    const double *T;
    const int32_t *top_k;
    const double *top_p, *min_p, *u;
    int64_t *tokens;
    double *vstar, *W, *cum;
    int64_t b0, b1;
    int status;
} icdf_job;

static void *icdf_worker(void *arg) {
    icdf_job *job = (icdf_job *)arg;
    entry *ent = (entry *)malloc(sizeof(entry) * (size_t)job->V);
    if (!ent) {
        job->status = TSAO_ERR_NOMEM;
        return NULL;
    }
    for (int64_t b = job->b0; b < job->b1; ++b) {
        const double *row = job->logits + b * job->stride;
        const int32_t *mrow = job->mask ? job->mask + b * job->mstride : NULL;
        double *cum = job->cum ? job->cum + b * job->V : NULL;
        row_result r;
        int st = sample_row(row, job->V, mrow, job->T[b], job->top_k[b], job->top_p[b],
                            job->min_p[b], 0, 0, 0, b, ent, &r, NULL, NULL);
        if (st != TSAO_OK) {
            job->status = st;
            break;
        }
        job->vstar[b] = r.vstar;
        job->W[b] = NAN;
        if (cum)
            for (int64_t i = 0; i < job->V; ++i) cum[i] = NAN;
        if (r.token < 0 || job->T[b] <= 0.0 || job->top_k[b] == 1) {
            job->tokens[b] = r.token; /* empty row, or greedy: the argmax */
            continue;
        }
        /* the kept tokens in index order, and their total weight */
        double W = 0.0;
        for (int64_t i = 0; i < job->V; ++i) {
            int allowed = mrow ? (int)(((uint32_t)mrow[i >> 5] >> (i & 31)) & 1u) : 1;
            if (!allowed || isinf(row[i]) || row[i] < r.vstar) continue;
            W += exp((row[i] - r.m) / job->T[b]);
            if (cum) cum[i] = W;
        }
        job->W[b] = W;
        double target = job->u[b] * W, S = 0.0;
        int64_t token = -1;
        for (int64_t i = 0; i < job->V; ++i) {
            int allowed = mrow ? (int)(((uint32_t)mrow[i >> 5] >> (i & 31)) & 1u) : 1;
            if (!allowed || isinf(row[i]) || row[i] < r.vstar) continue;
            S += exp((row[i] - r.m) / job->T[b]);
            token = i;
            if (S > target) break;
        }
        job->tokens[b] = token;
    }
    free(ent);
    return NULL;
}

int tsao_sample_icdf(const double *logits, int64_t B, int64_t V, int64_t stride,
                     const int32_t *mask, int64_t mstride, const double *T, const int32_t *top_k,
                     const double *top_p, const double *min_p, const double *u, int64_t *tokens,
                     double *vstar, double *W, double *cum, int nthreads) {
    if (B < 0 || V < 1 || stride < V || (mask && mstride < (V + 31) / 32)) return TSAO_ERR_ARG;
    for (int64_t b = 0; b < B; ++b)
        if (!(u[b] >= 0.0 && u[b] < 1.0)) return TSAO_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = (int)(B > 0 ? B : 1);
    icdf_job *jobs = (icdf_job *)calloc((size_t)nthreads, sizeof(icdf_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return TSAO_ERR_NOMEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        icdf_job *jb = &jobs[t];
        jb->logits = logits; jb->V = V; jb->stride = stride;
        jb->mask = mask; jb->mstride = mstride;
        jb->T = T; jb->top_k = top_k; jb->top_p = top_p; jb->min_p = min_p; jb->u = u;
        jb->tokens = tokens; jb->vstar = vstar; jb->W = W; jb->cum = cum;
        jb->b0 = B * t / nthreads;
        jb->b1 = B * (t + 1) / nthreads;
        jb->status = TSAO_OK;
    }
    int status = TSAO_OK;
    if (nthreads == 1) {
        icdf_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&th[t], NULL, icdf_worker, &jobs[t]) != 0) break;
            ++started;
        }
        for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
        for (int t = started; t < nthreads; ++t) icdf_worker(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != TSAO_OK) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}
