/*
 * CPU oracle for exact QSA block selection -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this file's library. It shares no code, header, table or helper with the
 * CUDA path; it is a plain, slow, FP64 restatement of what the selection
 * computes, written from the pages:
 *
 *  - "#3108 optimize exact QSA block scoring and top-k selection on gfx12",
 *    Summary items 1 and 4: a block score is the sum over the 4 query heads
 *    of the head's dot product with the block's summary key (the "4-head
 *    block score" assembled from per-head 32-lane reductions);
 *  - "#337 gfx12 QSA select", What items 1-2: only the batch's active blocks
 *    are scored and selected, never the capacity; the top-k is exact (the
 *    page reports selections equal to the reference in 256/256 queries),
 *    and an FP64 reference gates the scorer;
 *  - ties are broken by lower block id, and the selected ids are returned in
 *    ascending block-id order (reading taken where the pages are silent).
 *
 * Score (fp32 keys):  S[i][b] = sum_{h<4} sum_{d<128} q[i][h][d] * kblk[b][d]
 * in double precision: each head's dot product accumulates in natural d
 * order, and the heads are added in order 0..3. Every product of two floats
 * is exact in double, so S carries only the rounding of the additions.
 *
 * Score (int8 keys): the key element is kq8[b][d] * scale[b], scale an IEEE
 * binary16 value; the product (8-bit by 11-bit significands) is exact in
 * double, and the sum is formed exactly as above.
 *
 * Selection: sort the pairs (S, id) by S descending, then id ascending (a
 * strict total order), keep the first min(k, active) ids, sort them
 * ascending, and fill the remaining k - active slots (if any) with -1. A NaN
 * score counts as -infinity (so it ties with -inf and ranks below every
 * finite score); -0.0 and +0.0 compare equal (and so tie).
 *
 * Also here: the attention over the selected blocks' cells (FP64) and the
 * block summary keys (an fp32 restatement). The summary keys are "parity
 * unpinned" as to their definition: the pages time an append step but never
 * define how a block's key is built from its cells, so the function below is
 * a reading; its arithmetic is pinned, the definition is not.
 */
#include "qsa_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define QSA_H 4
#define QSA_D 128

int qsa_oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n < 1 ? 1 : (int)n;
}

/* ---- row-parallel driver (rows are independent) ---------------------- */

typedef void (*row_fn)(void *ctx, long row);

typedef struct {
    row_fn fn;
    void *ctx;
    long nrows;
    int tid, nthreads;
} row_job;

static void *row_worker(void *arg) {
    row_job *j = (row_job *)arg;
    for (long r = j->tid; r < j->nrows; r += j->nthreads) j->fn(j->ctx, r);
    return NULL;
}

static void for_each_row(row_fn fn, void *ctx, long nrows, int nthreads) {
    if (nthreads <= 0) nthreads = qsa_oracle_default_threads();
    if (nthreads > nrows) nthreads = (int)(nrows > 0 ? nrows : 1);
    if (nthreads == 1) {
        for (long r = 0; r < nrows; ++r) fn(ctx, r);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    row_job *jobs = (row_job *)malloc(sizeof(row_job) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].nrows = nrows;
        jobs[t].tid = t; jobs[t].nthreads = nthreads;
        pthread_create(&th[t], NULL, row_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
}

/* ---- IEEE 754 binary16 -> double (from the format's definition) ------- */

double qsa_oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)            v = ldexp((double)m, -24);                 /* zero / subnormal */
    else if (e == 0x1F)    v = (m == 0) ? INFINITY : NAN;             /* inf / NaN        */
    else                   v = ldexp((double)(1024 + m), e - 25);     /* normal           */
    return sign ? -v : v;
}

/* ---- block scores ----------------------------------------------------- */

typedef struct {
    const float *q;
    const float *kblk;
    const int8_t *kq8;
    const uint16_t *kscale;
    long active;
    double *S;
} score_ctx;

static void score_row_f32(void *vctx, long i) {
    const score_ctx *c = (const score_ctx *)vctx;
    const float *qi = c->q + (size_t)i * QSA_H * QSA_D;
    double *Si = c->S + (size_t)i * (size_t)c->active;
    for (long b = 0; b < c->active; ++b) {
        const float *kb = c->kblk + (size_t)b * QSA_D;
        double total = 0.0;
        for (int h = 0; h < QSA_H; ++h) {
            const float *qh = qi + h * QSA_D;
            double dot = 0.0;
            for (int d = 0; d < QSA_D; ++d) dot += (double)qh[d] * (double)kb[d];
            total += dot;
        }
        Si[b] = total;
    }
}

static void score_row_q8(void *vctx, long i) {
    const score_ctx *c = (const score_ctx *)vctx;
    const float *qi = c->q + (size_t)i * QSA_H * QSA_D;
    double *Si = c->S + (size_t)i * (size_t)c->active;
    for (long b = 0; b < c->active; ++b) {
        const int8_t *kb = c->kq8 + (size_t)b * QSA_D;
        double scale = qsa_oracle_half_to_double(c->kscale[b]);
        double total = 0.0;
        for (int h = 0; h < QSA_H; ++h) {
            const float *qh = qi + h * QSA_D;
            double dot = 0.0;
            for (int d = 0; d < QSA_D; ++d) dot += (double)qh[d] * ((double)kb[d] * scale);
            total += dot;
        }
        Si[b] = total;
    }
}

void qsa_oracle_scores(const float *q, const float *kblk, long nq, long active,
                       double *S, int nthreads) {
    score_ctx c = {q, kblk, NULL, NULL, active, S};
    for_each_row(score_row_f32, &c, nq, nthreads);
}

void qsa_oracle_scores_q8(const float *q, const int8_t *kq8, const uint16_t *kscale,
                          long nq, long active, double *S, int nthreads) {
    score_ctx c = {q, NULL, kq8, kscale, active, S};
    for_each_row(score_row_q8, &c, nq, nthreads);
}

/* ---- exact top-k by full sort ---------------------------------------- */

typedef struct { double s; int32_t id; } scored_id;

/* A NaN score counts as -infinity (it ties with -inf); -0.0 == +0.0. */
static double rank_value(double s) { return isnan(s) ? -INFINITY : s; }

/* Strict total order: higher score first, then lower id. */
static int by_score_desc_id_asc(const void *pa, const void *pb) {
    const scored_id *a = (const scored_id *)pa, *b = (const scored_id *)pb;
    double va = rank_value(a->s), vb = rank_value(b->s);
    if (va > vb) return -1;
    if (va < vb) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

static int by_id_asc(const void *pa, const void *pb) {
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

typedef struct {
    const double *S64;
    const float *S32;
    long active, k;
    int32_t *ids;
} topk_ctx;

static void topk_row(void *vctx, long i) {
    const topk_ctx *c = (const topk_ctx *)vctx;
    long n = c->active;
    scored_id *pairs = (scored_id *)malloc(sizeof(scored_id) * (size_t)(n > 0 ? n : 1));
    for (long b = 0; b < n; ++b) {
        pairs[b].s = c->S64 ? c->S64[(size_t)i * n + b] : (double)c->S32[(size_t)i * n + b];
        pairs[b].id = (int32_t)b;
    }
    qsort(pairs, (size_t)n, sizeof(scored_id), by_score_desc_id_asc);
    long m = c->k < n ? c->k : n;
    int32_t *out = c->ids + (size_t)i * (size_t)c->k;
    for (long j = 0; j < m; ++j) out[j] = pairs[j].id;
    qsort(out, (size_t)m, sizeof(int32_t), by_id_asc);
    for (long j = m; j < c->k; ++j) out[j] = -1;
    free(pairs);
}

void qsa_oracle_topk_f64(const double *S, long nq, long active, long k, int32_t *ids,
                         int nthreads) {
    topk_ctx c = {S, NULL, active, k, ids};
    for_each_row(topk_row, &c, nq, nthreads);
}

void qsa_oracle_topk_f32(const float *scores, long nq, long active, long k, int32_t *ids,
                         int nthreads) {
    topk_ctx c = {NULL, scores, active, k, ids};
    for_each_row(topk_row, &c, nq, nthreads);
}

/* ---- sparse attention over the selected blocks ------------------------ */
/*
 * Passages: "#3224 [Engine] perf(hip): tune RDNA4 QSA prompt WMMA path
 * (STRATA_HIP_WMMA stays opt-in)", Summary and Evidence section 2 (the QSA
 * attention reads int8 K and V cells, each with a binary16 scale, and is
 * gated against an FP64 host reference); "#3102 perf(hip): enable wave32 QSA
 * decode attention and MMVQ row reuse on gfx12", item D5 (decode attention
 * runs over the KV cells in chunks whose partial results are merged in the
 * chunks' sequential order).
 *
 * The pages name the kernels but print no formula; the readings taken:
 *  - query i attends the cells of the blocks listed in ids[i][0..k): block b
 *    holds cells 4b .. 4b+3 (those below ncells); a negative id, or one at or
 *    past the last block, is padding and contributes nothing; a listed block
 *    contributes once per listing;
 *  - cell c's key and value are kq[c][d] * ks[c] and vq[c][d] * vs[c] (int8
 *    times one IEEE binary16 scale per cell; both products exact in double);
 *  - the 4 query heads share the cells, as they share the block keys:
 *    logit[h][c] = (sum_d q[i][h][d] * key[c][d]) / sqrt(128);
 *  - out[i][h][d] = sum_c w[h][c] * value[c][d] with w[h][.] the softmax of
 *    logit[h][.] over the attended cells (the largest logit is subtracted
 *    before exponentiating, which leaves w unchanged);
 *  - a query with no attended cell gets out = 0.
 * Each product of a float with a key element is exact in double; the sums
 * run in the cells' listing order, then cell order within a block.
 */
typedef struct {
    const float *q;
    const int8_t *kq, *vq;
    const uint16_t *ks, *vs;
    long ncells, k;
    const int32_t *ids;
    double *out;
} attn_ctx;

static void attn_row(void *vctx, long i) {
    const attn_ctx *c = (const attn_ctx *)vctx;
    const long nblocks = (c->ncells + 3) / 4;
    double *o = c->out + (size_t)i * QSA_H * QSA_D;
    for (int e = 0; e < QSA_H * QSA_D; ++e) o[e] = 0.0;
    long *cells = (long *)malloc(sizeof(long) * (size_t)(4 * (c->k > 0 ? c->k : 1)));
    long n = 0;
    for (long j = 0; j < c->k; ++j) {
        const long b = c->ids[(size_t)i * (size_t)c->k + (size_t)j];
        if (b < 0 || b >= nblocks) continue;
        for (long t = 0; t < 4; ++t)
            if (4 * b + t < c->ncells) cells[n++] = 4 * b + t;
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    const double temperature = 1.0 / sqrt((double)QSA_D);
    for (int h = 0; h < QSA_H && n > 0; ++h) {
        const float *qh = c->q + ((size_t)i * QSA_H + (size_t)h) * QSA_D;
        double top = -INFINITY;
        for (long t = 0; t < n; ++t) {
            const int8_t *kc = c->kq + (size_t)cells[t] * QSA_D;
            const double scale = qsa_oracle_half_to_double(c->ks[cells[t]]);
            double dot = 0.0;
            for (int d = 0; d < QSA_D; ++d) dot += (double)qh[d] * ((double)kc[d] * scale);
            w[t] = dot * temperature;
            if (w[t] > top) top = w[t];
        }
        double total = 0.0;
        for (long t = 0; t < n; ++t) {
            w[t] = exp(w[t] - top);
            total += w[t];
        }
        for (long t = 0; t < n; ++t) {
            const int8_t *vc = c->vq + (size_t)cells[t] * QSA_D;
            const double scale = qsa_oracle_half_to_double(c->vs[cells[t]]);
            const double p = w[t] / total;
            for (int d = 0; d < QSA_D; ++d) o[h * QSA_D + d] += p * ((double)vc[d] * scale);
        }
    }
    free(w);
    free(cells);
}

void qsa_oracle_sparse_attn(const float *q, const int8_t *kq, const uint16_t *ks, const int8_t *vq,
                            const uint16_t *vs, long ncells, const int32_t *ids, long nq, long k,
                            double *out, int nthreads) {
    attn_ctx c = {q, kq, vq, ks, vs, ncells, k, ids, out};
    for_each_row(attn_row, &c, nq, nthreads);
}

/* ---- block summary keys ------------------------------------------------ */
/*
 * Passages: "#3108 optimize exact QSA block scoring and top-k selection on
 * gfx12", the Microbenchmark & Parity Evidence table (its decode layer times
 * "append + scores + topk + attn": a block's summary key is brought up to
 * date when cells are appended). The pages do not say how a key is built
 * from its cells; the reading taken:
 *  - block b's key is the element-wise mean of its present cells (cells
 *    4b .. 4b+3 below ncells), each cell being kq[c][d] * ks[c] (int8 times
 *    a binary16 scale; the product is exact in fp32);
 *  - the int8 form (the decode scorer's key format) has one binary16 scale
 *    per block, s = binary16(max_d |key[d]| / 127) rounded to nearest even,
 *    and codes rint(key[d] / s) (0 when s is 0);
 *  - a block with no present cell gets a zero key, zero codes, scale 0.
 * Because the integer codes are decided by float arithmetic, this restates
 * the computation in fp32, in one order: sum = ((0 + x0) + x1) + ... over the
 * present cells, key = sum / n, s32 = max / 127, each an IEEE single
 * operation (the products are exact, so contracting them into fused
 * multiply-adds changes nothing).
 */
static uint16_t float_to_half_rne(float f) {
    /* binary32 -> binary16, round to nearest even, from the formats'
     * definitions (no NaN or infinity arises here). */
    union { float f; uint32_t u; } v = {f};
    const uint32_t sign = (v.u >> 16) & 0x8000u;
    const uint32_t a = v.u & 0x7FFFFFFFu;
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);       /* rounds past 65504: infinity */
    const int e = (int)(a >> 23) - 127;                              /* unbiased exponent */
    if (e >= -14) {                                                  /* normal binary16 */
        uint32_t m = a & 0x7FFFFFu;                                  /* 23-bit fraction */
        uint32_t h = (uint32_t)(e + 15) << 10 | (m >> 13);
        const uint32_t rest = m & 0x1FFFu;                           /* the 13 dropped bits */
        if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;   /* may carry into the exponent */
        return (uint16_t)(sign | h);
    }
    /* subnormal binary16: value = k * 2^-24 with k = |f| * 2^24 rounded to
     * nearest even (k = 1024 is the smallest normal, whose encoding it is) */
    const double r = rint(fabs((double)f) * 16777216.0);
    return (uint16_t)(sign | (uint16_t)r);
}

uint16_t qsa_oracle_float_to_half(float f) { return float_to_half_rne(f); }

void qsa_oracle_block_summary(const int8_t *kq, const uint16_t *ks, long ncells, long b0, long b1,
                              float *key, int8_t *kq8, uint16_t *kscale) {
    for (long b = b0; b < b1; ++b) {
        long n = ncells - 4 * b;
        if (n > 4) n = 4;
        if (n < 0) n = 0;
        float mean[QSA_D];
        for (int d = 0; d < QSA_D; ++d) {
            float sum = 0.0f;
            for (long t = 0; t < n; ++t) {
                const long c = 4 * b + t;
                const float x = (float)kq[(size_t)c * QSA_D + d] * (float)qsa_oracle_half_to_double(ks[c]);
                sum = sum + x;
            }
            mean[d] = n > 0 ? sum / (float)n : 0.0f;
        }
        const size_t row = (size_t)(b - b0);
        if (key != NULL)
            for (int d = 0; d < QSA_D; ++d) key[row * QSA_D + d] = mean[d];
        if (kq8 != NULL) {
            float top = 0.0f;
            for (int d = 0; d < QSA_D; ++d) top = fmaxf(top, fabsf(mean[d]));
            const uint16_t sh = float_to_half_rne(top / 127.0f);
            const float s = (float)qsa_oracle_half_to_double(sh);
            kscale[row] = sh;
            for (int d = 0; d < QSA_D; ++d) {
                float c = s > 0.0f ? rintf(mean[d] / s) : 0.0f;
                if (c > 127.0f) c = 127.0f;
                if (c < -127.0f) c = -127.0f;
                kq8[row * QSA_D + d] = (int8_t)c;
            }
        }
    }
}
