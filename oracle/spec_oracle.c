/*
 * spec_oracle.c -- plain, slow, obviously-correct CPU oracle for ragged
 * speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library; both are written
 * separately from the same definitions.
 *
 * Everything is computed in double precision from the exact input values
 * (bf16 and fp32 convert exactly to double).  Ranks use a full sort.  No
 * blocking, fusion or reordering beyond the definitions below.
 *
 * Sources (web pages; section names as printed there):
 *   [vSpec]  "vllm-hust-vSpec" README (PyPI PKG-INFO of vllm_hust_vspec 0.13.0):
 *            §"支持范围" (relaxed top-K acceptance), §"EAGLE 功能" (strict
 *            greedy top-1 acceptance, relaxed top-K with strict prefix, no
 *            per-request D2H in acceptance), §"代码所有权".
 *   [xLLM]   xLLM docs "自适应投机推理" (adaptive speculative inference):
 *            §"自适应 draft 步长（MTP）" (per-position prefix acceptance and
 *            the objective B*(1+sum(prefix_acceptance[:k]))/cost_ms),
 *            §"基于 MTP logits 的自适应 target 验证" (confidence
 *            exp(selected_logit - logsumexp(draft_logits)), device-side prefix
 *            allocation and packing with device offsets),
 *            §"启动示例" (ragged rejection sampler over packed rows with
 *            per-request parameters via packed-row owners; point-mass draft:
 *            accept while the sample equals the draft, first mismatching
 *            sample is the replacement, last row's sample is the bonus;
 *            temperature 0 is greedy; top-k/top-p/min-p follow the ordinary
 *            sampler).
 *   [Philox] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *            1, 2, 3", SC'11 -- the Philox4x32 bijection with 10 rounds.
 *
 * Readings where the pages are silent:
 *   - argmax ties: lowest index; -0.0 equals +0.0.
 *   - filter order: temperature, then top-k and min-p as value thresholds
 *     (they commute), then top-p over their survivors; ties at a threshold
 *     are kept or cut as whole groups.
 *   - sampling: Gumbel-max over the survivors with one Philox uniform per
 *     vocabulary index (key = seed, counter = (i>>2, position, request, step),
 *     word i&3), u = (2*(x>>9)+1) * 2^-24, g = -log(-log u).
 *   - prefix allocation: cumulative product of confidences >= threshold,
 *     optional global row budget keeps the top (G-B) entries ordered by
 *     (cumulative confidence desc, request asc, position asc).
 *   - NaN and +inf logits are outside the contract; -inf is allowed.
 *   - confidence margin: the gap max - z[d] is taken in fp32 (the inputs
 *     are exact fp32 values); position j of request b is eligible when
 *     j >= from_position and generated[b] + j >= after_tokens.
 *
 * Parity pins for every function live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* status bits reported by the verify functions (the documented contract) */
#define OR_BAD_TEMPERATURE 0x1u
#define OR_BAD_TOP_K       0x2u
#define OR_BAD_TOP_P       0x4u
#define OR_BAD_MIN_P       0x8u
#define OR_BAD_ROWS        0x10u
#define OR_BAD_SELECTED    0x20u
#define OR_BAD_RELAXED_K   0x40u
#define OR_BAD_BUDGET      0x80u
#define OR_BAD_MARGIN      0x200u

/* ------------------------------------------------------------------------ */
/* threads                                                                  */
/* ------------------------------------------------------------------------ */

int oracle_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* input decoding                                                           */
/* ------------------------------------------------------------------------ */

/* dtype 0 = fp32, 1 = bf16 (stored as the upper 16 bits of an fp32). */
static double logit_at(const void *base, int dtype, int64_t ld, int64_t r, int64_t i)
{
    if (dtype == 0)
        return (double)((const float *)base)[r * ld + i];
    uint32_t u = (uint32_t)((const uint16_t *)base)[r * ld + i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void load_row(const void *base, int dtype, int64_t ld, int32_t V, int64_t r, double *z)
{
    for (int32_t i = 0; i < V; ++i)
        z[i] = logit_at(base, dtype, ld, r, i);
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 [Philox]                                                   */
/* ------------------------------------------------------------------------ */

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        /* two 32x32->64 products; the high halves are mixed with the
           other two counter words and the round key, the low halves move */
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        /* Weyl key schedule: golden ratio and sqrt(3)-1 */
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* 32 random bits -> uniform in (0,1): the top 23 bits, centred in their cell */
double oracle_uniform(uint32_t x)
{
    return (2.0 * (double)(x >> 9) + 1.0) * ldexp(1.0, -24);
}

/* uniform draw for vocabulary index i at (seed, request, position, step) */
double oracle_token_uniform(uint64_t seed, uint32_t rid, uint32_t pos, uint32_t step, uint32_t i)
{
    uint32_t ctr[4] = { i >> 2, pos, rid, step };
    uint32_t key[2] = { (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32) };
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return oracle_uniform(out[i & 3u]);
}

/* ------------------------------------------------------------------------ */
/* A1: max / first argmax / log-sum-exp of one row                          */
/* ------------------------------------------------------------------------ */

static void reduce_row(const double *z, int32_t V, double *mx, double *lse, int32_t *amax)
{
    double m = -INFINITY;
    int32_t a = 0;
    for (int32_t i = 0; i < V; ++i)
        if (z[i] > m) { m = z[i]; a = i; }        /* strict: first index wins */
    double l;
    if (m == -INFINITY || V == 0) {
        l = -INFINITY;
    } else {
        double s = 0.0;
        for (int32_t i = 0; i < V; ++i)
            s += exp(z[i] - m);
        l = m + log(s);
    }
    if (mx) *mx = m;
    if (lse) *lse = l;
    if (amax) *amax = a;
}

void oracle_row_reduce(const void *logits, int dtype, int64_t ld, int32_t V, int32_t R,
                       double *row_max, double *row_lse, int32_t *row_argmax)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < R; ++r) {
        double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
        load_row(logits, dtype, ld, V, r, z);
        reduce_row(z, V, row_max ? &row_max[r] : NULL, row_lse ? &row_lse[r] : NULL,
                   row_argmax ? &row_argmax[r] : NULL);
        free(z);
    }
}

/* ------------------------------------------------------------------------ */
/* ragged rows                                                              */
/* ------------------------------------------------------------------------ */

/* k_b of request b, or -1 if its row range is not a valid request */
static int32_t request_k(const int32_t *cu_rows, int32_t b, int32_t k_max)
{
    int32_t n = cu_rows[b + 1] - cu_rows[b];
    if (cu_rows[0] != 0 || n < 1 || n - 1 > k_max)
        return -1;
    return n - 1;
}

/* Emit the accepted draft prefix followed by one target token (the
   replacement at the first rejection, or the bonus after a full accept). */
static void emit(int32_t b, int32_t k_max, int32_t a, const int32_t *drafts, int32_t tok,
                 int32_t *accepted_len, int32_t *out_tokens, int32_t *next_token)
{
    accepted_len[b] = a;
    next_token[b] = tok;
    for (int32_t j = 0; j <= k_max; ++j) {
        int32_t v = -1;
        if (j < a) v = drafts[j];
        else if (j == a) v = tok;
        out_tokens[(int64_t)b * (k_max + 1) + j] = v;
    }
}

static void emit_invalid(int32_t b, int32_t k_max, int32_t *accepted_len, int32_t *out_tokens,
                         int32_t *next_token)
{
    accepted_len[b] = 0;
    next_token[b] = -1;
    for (int32_t j = 0; j <= k_max; ++j)
        out_tokens[(int64_t)b * (k_max + 1) + j] = -1;
}

/* owner request of packed row r (rows of invalid requests have no owner) */
static void row_owners(const int32_t *cu_rows, int32_t B, int32_t k_max, int32_t *owner, int32_t *pos)
{
    for (int32_t b = 0; b < B; ++b) {
        if (request_k(cu_rows, b, k_max) < 0)
            continue;
        for (int32_t r = cu_rows[b]; r < cu_rows[b + 1]; ++r) {
            owner[r] = b;
            pos[r] = r - cu_rows[b];
        }
    }
}

static int32_t total_rows_of(const int32_t *cu_rows, int32_t B)
{
    int32_t R = cu_rows[B];
    return R > 0 ? R : 0;
}

/* ------------------------------------------------------------------------ */
/* A2: greedy verification                                                  */
/* ------------------------------------------------------------------------ */

uint32_t oracle_verify_greedy(const void *logits, int dtype, int64_t ld, int32_t V,
                              int32_t B, int32_t k_max, const int32_t *cu_rows,
                              const int32_t *draft_ids,
                              int32_t *accepted_len, int32_t *out_tokens, int32_t *next_token,
                              double *row_max, double *row_lse, int32_t *row_argmax)
{
    uint32_t status = 0;
    int32_t R = total_rows_of(cu_rows, B);
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    double *mx = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
    double *ls = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
    oracle_row_reduce(logits, dtype, ld, V, R, mx, ls, amax);
    for (int32_t b = 0; b < B; ++b) {
        int32_t k = request_k(cu_rows, b, k_max);
        if (k < 0) { status |= OR_BAD_ROWS; emit_invalid(b, k_max, accepted_len, out_tokens, next_token); continue; }
        const int32_t r0 = cu_rows[b];
        /* longest prefix of drafts equal to the target's top token */
        int32_t a = 0;
        while (a < k && draft_ids[r0 + a] == amax[r0 + a])
            ++a;
        emit(b, k_max, a, &draft_ids[r0], amax[r0 + a], accepted_len, out_tokens, next_token);
    }
    for (int32_t r = 0; r < R; ++r) {
        if (row_max) row_max[r] = mx[r];
        if (row_lse) row_lse[r] = ls[r];
        if (row_argmax) row_argmax[r] = amax[r];
    }
    free(amax); free(mx); free(ls);
    return status;
}

/* ------------------------------------------------------------------------ */
/* A3: filtered sampling of one row                                         */
/* ------------------------------------------------------------------------ */

typedef struct { double v; int32_t i; } ranked;

static int by_value_desc(const void *pa, const void *pb)
{
    const ranked *a = (const ranked *)pa, *b = (const ranked *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

/*
 * Survivor set of the temperature / top-k / min-p / top-p filters (T > 0).
 * keep[i] = 1 for survivors.  *margin receives the smallest relative distance
 * of any floating-point threshold decision from its boundary (INFINITY when no
 * float decision was taken); disagreements with a float32 implementation can
 * only occur where this is tiny.
 */
void oracle_filter_row(const double *z, int32_t V, double T, int32_t top_k, double top_p,
                       double min_p, uint8_t *keep, double *margin)
{
    double m = -INFINITY;
    for (int32_t i = 0; i < V; ++i)
        if (z[i] > m) m = z[i];
    double mg = INFINITY;
    for (int32_t i = 0; i < V; ++i)
        keep[i] = 1;

    ranked *s = (ranked *)malloc(sizeof(ranked) * (size_t)(V > 0 ? V : 1));
    for (int32_t i = 0; i < V; ++i) { s[i].v = z[i]; s[i].i = i; }
    qsort(s, (size_t)V, sizeof(ranked), by_value_desc);

    /* top-k: keep i iff fewer than top_k values are strictly larger, i.e.
       z[i] >= the top_k-th largest value (ties at the threshold kept) */
    if (top_k > 0 && top_k < V) {
        double thr = s[top_k - 1].v;
        for (int32_t i = 0; i < V; ++i)
            if (z[i] < thr) keep[i] = 0;
    }
    /* min-p: keep i iff p_i / p_max = exp((z_i - max)/T) >= min_p */
    if (min_p > 0.0) {
        for (int32_t i = 0; i < V; ++i) {
            double ratio = exp((z[i] - m) / T);
            double d = fabs(ratio - min_p) / min_p;
            if (d < mg) mg = d;
            if (ratio < min_p) keep[i] = 0;
        }
    }
    /* top-p over the survivors S: keep i iff the mass of survivors with a
       strictly larger value is below top_p * (mass of S); whole tie groups */
    if (top_p < 1.0) {
        double W = 0.0;
        for (int32_t i = 0; i < V; ++i)
            if (keep[i]) W += exp((z[i] - m) / T);
        double above = 0.0;
        int32_t g = 0;
        int cut = 0;
        while (g < V) {
            int32_t h = g;
            while (h < V && s[h].v == s[g].v) ++h;       /* tie group [g, h) */
            double mass = 0.0;
            int any = 0;
            for (int32_t q = g; q < h; ++q)
                if (keep[s[q].i]) { mass += exp((s[q].v - m) / T); any = 1; }
            if (any) {
                if (!cut) {
                    double d = fabs(above - top_p * W) / W;
                    if (d < mg) mg = d;
                    if (above < top_p * W) above += mass;
                    else cut = 1;
                }
                if (cut)
                    for (int32_t q = g; q < h; ++q) keep[s[q].i] = 0;
            }
            g = h;
        }
    }
    free(s);
    if (margin) *margin = mg;
}

/*
 * Sampled token of one row.  T == 0 (or an all -inf row) gives the first
 * argmax.  Otherwise Gumbel-max over the survivors:
 *   y = argmax_{i in F} ( z_i / T - log(-log u_i) ),  lowest index on ties.
 * *margin_gumbel = gap between the best and second-best score.
 */
int32_t oracle_sample_row(const double *z, int32_t V, double T, int32_t top_k, double top_p,
                          double min_p, uint64_t seed, uint32_t rid, uint32_t pos, uint32_t step,
                          uint8_t *keep_out, double *margin_filter, double *margin_gumbel)
{
    double m; int32_t amax;
    reduce_row(z, V, &m, NULL, &amax);
    if (margin_filter) *margin_filter = INFINITY;
    if (margin_gumbel) *margin_gumbel = INFINITY;
    if (!(T > 0.0) || m == -INFINITY) {
        if (keep_out) for (int32_t i = 0; i < V; ++i) keep_out[i] = (uint8_t)(i == amax);
        return amax;
    }
    uint8_t *keep = keep_out ? keep_out : (uint8_t *)malloc((size_t)(V > 0 ? V : 1));
    oracle_filter_row(z, V, T, top_k, top_p, min_p, keep, margin_filter);
    double best = -INFINITY, second = -INFINITY;
    int32_t y = -1;
    for (int32_t i = 0; i < V; ++i) {
        if (!keep[i]) continue;
        double u = oracle_token_uniform(seed, rid, pos, step, (uint32_t)i);
        double score = z[i] / T - log(-log(u));
        if (y < 0 || score > best) { second = best; best = score; y = i; }
        else if (score > second) second = score;
    }
    if (margin_gumbel) *margin_gumbel = best - second;
    if (!keep_out) free(keep);
    return y < 0 ? amax : y;
}

/* parameter validation shared by the stochastic verifier (the contract) */
static void sanitize(double *T, int32_t *top_k, double *top_p, double *min_p, uint32_t *status)
{
    if (!(*T >= 0.0) || isinf(*T)) { *status |= OR_BAD_TEMPERATURE; *T = 0.0; }
    if (*top_k < 0) { *status |= OR_BAD_TOP_K; *top_k = 0; }
    if (!(*top_p > 0.0 && *top_p <= 1.0)) { *status |= OR_BAD_TOP_P; *top_p = 1.0; }
    if (!(*min_p >= 0.0 && *min_p <= 1.0)) { *status |= OR_BAD_MIN_P; *min_p = 0.0; }
}

/* ------------------------------------------------------------------------ */
/* A3 + A4: stochastic verification with a point-mass draft                 */
/* ------------------------------------------------------------------------ */

uint32_t oracle_verify_sample(const void *logits, int dtype, int64_t ld, int32_t V,
                              int32_t B, int32_t k_max, const int32_t *cu_rows,
                              const int32_t *draft_ids,
                              const float *temperature, const int32_t *top_k,
                              const float *top_p, const float *min_p,
                              const uint64_t *seed, const uint32_t *request_id, uint32_t step,
                              int32_t *accepted_len, int32_t *out_tokens, int32_t *next_token,
                              int32_t *row_token, double *row_margin_filter,
                              double *row_margin_gumbel)
{
    uint32_t status = 0;
    int32_t R = total_rows_of(cu_rows, B);
    int32_t n = R > 0 ? R : 1;
    int32_t *owner = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *y = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    for (int32_t r = 0; r < R; ++r) { owner[r] = -1; pos[r] = 0; y[r] = -1; }
    row_owners(cu_rows, B, k_max, owner, pos);

    for (int32_t b = 0; b < B; ++b) {
        double T = temperature[b], tp = top_p[b], mp = min_p[b];
        int32_t tk = top_k[b];
        if (request_k(cu_rows, b, k_max) >= 0)
            sanitize(&T, &tk, &tp, &mp, &status);
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < R; ++r) {
        int32_t b = owner[r];
        if (b < 0) continue;
        double T = temperature[b], tp = top_p[b], mp = min_p[b];
        int32_t tk = top_k[b];
        uint32_t ignored = 0;
        sanitize(&T, &tk, &tp, &mp, &ignored);
        uint32_t rid = request_id ? request_id[b] : (uint32_t)b;
        double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
        load_row(logits, dtype, ld, V, r, z);
        double mf, mgb;
        y[r] = oracle_sample_row(z, V, T, tk, tp, mp, seed[b], rid, (uint32_t)pos[r], step,
                                 NULL, &mf, &mgb);
        if (row_margin_filter) row_margin_filter[r] = mf;
        if (row_margin_gumbel) row_margin_gumbel[r] = mgb;
        free(z);
    }

    for (int32_t b = 0; b < B; ++b) {
        int32_t k = request_k(cu_rows, b, k_max);
        if (k < 0) { status |= OR_BAD_ROWS; emit_invalid(b, k_max, accepted_len, out_tokens, next_token); continue; }
        const int32_t r0 = cu_rows[b];
        /* accept while the sampled target token equals the draft token */
        int32_t a = 0;
        while (a < k && y[r0 + a] == draft_ids[r0 + a])
            ++a;
        emit(b, k_max, a, &draft_ids[r0], y[r0 + a], accepted_len, out_tokens, next_token);
    }
    if (row_token)
        for (int32_t r = 0; r < R; ++r) row_token[r] = y[r];
    free(owner); free(pos); free(y);
    return status;
}

/* ------------------------------------------------------------------------ */
/* A5: relaxed top-K acceptance with strict prefix [vSpec]                  */
/* ------------------------------------------------------------------------ */

uint32_t oracle_verify_relaxed(const void *logits, int dtype, int64_t ld, int32_t V,
                               int32_t B, int32_t k_max, const int32_t *cu_rows,
                               const int32_t *draft_ids, const int32_t *relaxed_k,
                               int32_t *accepted_len, int32_t *out_tokens, int32_t *next_token,
                               int32_t *row_argmax, int32_t *row_rank)
{
    uint32_t status = 0;
    int32_t R = total_rows_of(cu_rows, B);
    int32_t n = R > 0 ? R : 1;
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *rank = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);

#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < R; ++r) {
        double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
        load_row(logits, dtype, ld, V, r, z);
        reduce_row(z, V, NULL, NULL, &amax[r]);
        /* rank of the draft token: number of strictly larger logits;
           out-of-vocabulary drafts get rank V (never accepted) */
        int32_t d = draft_ids[r];
        int32_t cnt = V;
        if (d >= 0 && d < V) {
            cnt = 0;
            for (int32_t i = 0; i < V; ++i)
                if (z[i] > z[d]) ++cnt;
        }
        rank[r] = cnt;
        free(z);
    }
    for (int32_t b = 0; b < B; ++b) {
        int32_t k = request_k(cu_rows, b, k_max);
        if (k < 0) { status |= OR_BAD_ROWS; emit_invalid(b, k_max, accepted_len, out_tokens, next_token); continue; }
        int32_t K = relaxed_k[b];
        if (K < 1) { status |= OR_BAD_RELAXED_K; K = 1; }
        const int32_t r0 = cu_rows[b];
        /* accept d_j iff it is among the target's top-K values (ties
           included); acceptance stops at the first failure */
        int32_t a = 0;
        while (a < k && rank[r0 + a] < K)
            ++a;
        emit(b, k_max, a, &draft_ids[r0], amax[r0 + a], accepted_len, out_tokens, next_token);
    }
    for (int32_t r = 0; r < R; ++r) {
        if (row_argmax) row_argmax[r] = amax[r];
        if (row_rank) row_rank[r] = rank[r];
    }
    free(amax); free(rank);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Greedy verification over an active vocabulary [vSpec §"EAGLE 功能",      */
/* §"代码所有权": active-vocabulary LM head with a full token-id map]        */
/* ------------------------------------------------------------------------ */

/* The target scores only V active columns; column i stands for the full
   token id vocab_ids[i].  The row's token is the full id of its first
   argmax column; drafts are full ids and are accepted while they equal it.
   row_argmax[r] is the column, row_token[r] the full id. */
uint32_t oracle_verify_greedy_active(const void *logits, int dtype, int64_t ld, int32_t V,
                                     int32_t B, int32_t k_max, const int32_t *cu_rows,
                                     const int32_t *draft_ids, const int32_t *vocab_ids,
                                     int32_t *accepted_len, int32_t *out_tokens,
                                     int32_t *next_token, int32_t *row_argmax,
                                     int32_t *row_token)
{
    uint32_t status = 0;
    int32_t R = total_rows_of(cu_rows, B);
    int32_t n = R > 0 ? R : 1;
    int32_t *col = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    oracle_row_reduce(logits, dtype, ld, V, R, NULL, NULL, col);
    for (int32_t r = 0; r < R; ++r)
        tok[r] = vocab_ids[col[r]];
    for (int32_t b = 0; b < B; ++b) {
        int32_t k = request_k(cu_rows, b, k_max);
        if (k < 0) { status |= OR_BAD_ROWS; emit_invalid(b, k_max, accepted_len, out_tokens, next_token); continue; }
        const int32_t r0 = cu_rows[b];
        int32_t a = 0;
        while (a < k && draft_ids[r0 + a] == tok[r0 + a])
            ++a;
        emit(b, k_max, a, &draft_ids[r0], tok[r0 + a], accepted_len, out_tokens, next_token);
    }
    for (int32_t r = 0; r < R; ++r) {
        if (row_argmax) row_argmax[r] = col[r];
        if (row_token) row_token[r] = tok[r];
    }
    free(col); free(tok);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Confidence-margin acceptance [vSpec §"启动", §"通用参数"]                  */
/* ------------------------------------------------------------------------ */

static int is_protected(int32_t d, const int32_t *ids, int32_t n)
{
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] == d) return 1;
    return 0;
}

/* Greedy acceptance loosened by a logit margin: a draft is accepted when it
   is the target's first argmax, or -- at an eligible position, for a token
   outside the protected set -- when its logit lies within margin[b] of the
   row maximum.  The prefix stays strict and the emitted token of the first
   rejected row (or the bonus row) is that row's first argmax, as in greedy
   verification.  row_ok[r] = 1 where the draft of row r passes. */
uint32_t oracle_verify_margin(const void *logits, int dtype, int64_t ld, int32_t V,
                              int32_t B, int32_t k_max, const int32_t *cu_rows,
                              const int32_t *draft_ids, const float *margin,
                              const int32_t *generated, int32_t from_position,
                              int32_t after_tokens, const int32_t *protected_ids,
                              int32_t n_protected,
                              int32_t *accepted_len, int32_t *out_tokens, int32_t *next_token,
                              int32_t *row_argmax, int32_t *row_ok)
{
    uint32_t status = 0;
    int32_t R = total_rows_of(cu_rows, B);
    int32_t n = R > 0 ? R : 1;
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    double *mx = (double *)malloc(sizeof(double) * (size_t)n);
    int32_t *ok = (int32_t *)calloc((size_t)n, sizeof(int32_t));
    oracle_row_reduce(logits, dtype, ld, V, R, mx, NULL, amax);
    for (int32_t b = 0; b < B; ++b) {
        int32_t k = request_k(cu_rows, b, k_max);
        if (k < 0) { status |= OR_BAD_ROWS; emit_invalid(b, k_max, accepted_len, out_tokens, next_token); continue; }
        float mg = margin[b];
        if (isnan(mg)) status |= OR_BAD_MARGIN;
        const int32_t r0 = cu_rows[b];
        const int32_t gen = generated ? generated[b] : 0;
        for (int32_t j = 0; j < k; ++j) {
            const int32_t r = r0 + j, d = draft_ids[r];
            if (d < 0 || d >= V) continue;
            if (d == amax[r]) { ok[r] = 1; continue; }
            if (isnan(mg) || j < from_position || (int64_t)gen + j < (int64_t)after_tokens) continue;
            if (is_protected(d, protected_ids, n_protected)) continue;
            /* both values are exact in fp32; the gap is rounded to fp32 */
            const float m32 = (float)mx[r];
            const float zd = (float)logit_at(logits, dtype, ld, r, d);
            const float gap = m32 - zd;
            if (gap <= mg) ok[r] = 1;
        }
        int32_t a = 0;
        while (a < k && ok[r0 + a])
            ++a;
        emit(b, k_max, a, &draft_ids[r0], amax[r0 + a], accepted_len, out_tokens, next_token);
    }
    for (int32_t r = 0; r < R; ++r) {
        if (row_argmax) row_argmax[r] = amax[r];
        if (row_ok) row_ok[r] = ok[r];
    }
    free(amax); free(mx); free(ok);
    return status;
}

/* ------------------------------------------------------------------------ */
/* A6 + A7: draft confidence, prefix-budget allocation and packing [xLLM]   */
/* ------------------------------------------------------------------------ */

typedef struct { double c; int32_t b, j; } entry;

static int by_conf_desc(const void *pa, const void *pb)
{
    const entry *a = (const entry *)pa, *b = (const entry *)pb;
    if (a->c > b->c) return -1;
    if (a->c < b->c) return 1;
    if (a->b != b->b) return a->b < b->b ? -1 : 1;
    return (a->j > b->j) - (a->j < b->j);
}

uint32_t oracle_draft_confidence(const void *draft_logits, int dtype, int64_t ld, int32_t V,
                                 int32_t B, int32_t k, const int32_t *selected,
                                 double threshold, int32_t max_rows,
                                 double *conf, int32_t *k_alloc, int32_t *cu_rows,
                                 int32_t *row_owner, int32_t *row_pos, int32_t *packed_draft,
                                 int32_t *total_rows, double *margin)
{
    uint32_t status = 0;
    int32_t Q = B * k;
    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Q > 0 ? Q : 1));
    uint32_t *bad = (uint32_t *)calloc((size_t)(Q > 0 ? Q : 1), sizeof(uint32_t));

    /* confidence of draft position (b, j): exp(selected - logsumexp(row)) */
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t q = 0; q < Q; ++q) {
        double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
        load_row(draft_logits, dtype, ld, V, q, z);
        double lse; int32_t amax;
        reduce_row(z, V, NULL, &lse, &amax);
        int32_t s = selected ? selected[q] : amax;
        tok[q] = s;
        if (s < 0 || s >= V) { conf[q] = 0.0; bad[q] = 1; }
        else conf[q] = exp(z[s] - lse);
        free(z);
    }
    for (int32_t q = 0; q < Q; ++q)
        if (bad[q]) status |= OR_BAD_SELECTED;

    /* cumulative confidence c_{b,j} = prod_{i<=j} conf[b][i]; the number of
       positions whose cumulative confidence reaches the threshold */
    double *cum = (double *)malloc(sizeof(double) * (size_t)(Q > 0 ? Q : 1));
    double mg = INFINITY;
    int32_t want = 0;
    for (int32_t b = 0; b < B; ++b) {
        double c = 1.0;
        int32_t cnt = 0;
        for (int32_t j = 0; j < k; ++j) {
            c *= conf[b * k + j];
            cum[b * k + j] = c;
            if (c >= threshold) ++cnt;
            if (threshold > 0.0) {
                double d = fabs(c - threshold) / threshold;
                if (d < mg) mg = d;
            }
        }
        k_alloc[b] = cnt;
        want += cnt + 1;
    }

    /* optional global row budget G: keep the best (G - B) draft positions */
    if (max_rows > 0 && want > max_rows) {
        if (max_rows < B) {
            status |= OR_BAD_BUDGET;
        } else {
            int32_t n = want - B;
            entry *e = (entry *)malloc(sizeof(entry) * (size_t)(n > 0 ? n : 1));
            int32_t w = 0;
            for (int32_t b = 0; b < B; ++b)
                for (int32_t j = 0; j < k_alloc[b]; ++j) {
                    e[w].c = cum[b * k + j]; e[w].b = b; e[w].j = j; ++w;
                }
            qsort(e, (size_t)n, sizeof(entry), by_conf_desc);
            int32_t keep = max_rows - B;
            for (int32_t b = 0; b < B; ++b) k_alloc[b] = 0;
            for (int32_t q = 0; q < keep; ++q) k_alloc[e[q].b] += 1;
            if (keep > 0 && keep < n && e[keep - 1].c > 0.0) {
                double d = (e[keep - 1].c - e[keep].c) / e[keep - 1].c;
                if (d < mg) mg = d;
            }
            free(e);
        }
    }

    /* packing: exclusive scan of (k_b + 1) and per-row owner / position */
    cu_rows[0] = 0;
    for (int32_t b = 0; b < B; ++b)
        cu_rows[b + 1] = cu_rows[b] + k_alloc[b] + 1;
    int32_t R = cu_rows[B];
    int32_t cap = B * (k + 1);
    for (int32_t r = 0; r < cap; ++r) {
        row_owner[r] = -1; row_pos[r] = -1;
        if (packed_draft) packed_draft[r] = -1;
    }
    for (int32_t b = 0; b < B; ++b)
        for (int32_t j = 0; j <= k_alloc[b]; ++j) {
            int32_t r = cu_rows[b] + j;
            row_owner[r] = b;
            row_pos[r] = j;
            if (packed_draft) packed_draft[r] = j < k_alloc[b] ? tok[b * k + j] : -1;
        }
    if (total_rows) *total_rows = R;
    if (margin) *margin = mg;
    free(tok); free(bad); free(cum);
    return status;
}

/* ------------------------------------------------------------------------ */
/* A8: per-position prefix-acceptance counters [xLLM]                       */
/* ------------------------------------------------------------------------ */

/* acc[j] += #{b : a_b > j}, ver[j] += #{b : k_b > j}, hist[a_b] += 1.
   prefix_acceptance[j] = acc[j] / ver[j].  Requests with invalid rows are
   skipped. */
uint32_t oracle_prefix_stats(const int32_t *accepted_len, const int32_t *cu_rows, int32_t B,
                             int32_t k_max, int64_t *acc, int64_t *ver, int64_t *hist)
{
    uint32_t status = 0;
    for (int32_t b = 0; b < B; ++b) {
        int32_t k = request_k(cu_rows, b, k_max);
        int32_t a = accepted_len[b];
        if (k < 0 || a < 0 || a > k) { status |= OR_BAD_ROWS; continue; }
        for (int32_t j = 0; j < k_max; ++j) {
            if (a > j) acc[j] += 1;
            if (k > j) ver[j] += 1;
        }
        if (hist) hist[a] += 1;
    }
    return status;
}
