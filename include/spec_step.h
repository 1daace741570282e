/*
 * spec_step.h -- C ABI of libspecverify's adaptive draft-step controller:
 * the host-side choice of one speculative step count k for the next decode
 * batch from the prefix-acceptance counters of completed verifications.
 *
 * What it computes (xLLM docs "自适应投机推理" (adaptive speculative
 * inference); section names as printed on the page):
 *   §"自适应 draft 步长（MTP）": before each batch the engine picks one k for
 *     the whole batch, up to the maximum step count, maximising
 *       score(k) = B * (1 + sum_{j<k} prefix_acceptance[j]) / cost_ms(k),
 *     from per-position prefix acceptance of completed batches and the
 *     full-step cost of each candidate k.
 *   §"可选的步长配置文件": the acceptance window (20 completed batches), the
 *     re-scoring interval (every 5 completed batches) and the minimum
 *     predicted relative gain to switch (0.05, to be strictly exceeded).
 *   §"成本模型与覆盖范围": full-step cost models -- an SPS table over the
 *     physical target graph rows G (cost 1000 / SPS(G) ms) or an additive
 *     fit bias + alpha(Bcap) + theta(G) seconds over the physical request
 *     bucket Bcap and G; G is the first captured bucket covering the rows a
 *     step verifies, B * (k + 1) (the page's example: B = 8 with 5 drafts
 *     binds G = 8, 16, 32, 48 for k = 0, 1, 3, 5).
 *
 * Readings where the page is silent:
 *   - prefix_acceptance[j] = sum over the window of acc[j] / sum of ver[j],
 *     with acc[j] = #(accepted length > j) and ver[j] = #(draft length > j)
 *     per batch: the A8 counters of the verify calls.
 *   - Positions never verified in the window (beyond the largest k used)
 *     are extrapolated with the conditional acceptance of the last verified
 *     position, pa[L] / pa[L-1] (pa[0] when L = 0), clamped to [0, 1]: the
 *     i.i.d. acceptance model.  Without it a smaller k could never grow.
 *   - Ties in score go to the smaller k; a switch needs
 *     score(best) > (1 + switch_min_gain) * score(current); an infeasible
 *     current k (cost +inf) scores 0, so any feasible k replaces it.
 *   - An empty window (no verified position yet) keeps the current k.
 *
 * Conventions: every pointer is HOST memory owned by the caller; nothing is
 * allocated; no CUDA call is made, so these run without a GPU.  Return values
 * are spec_result codes; an invalid argument returns SPEC_ERR_INVALID_ARG
 * with the state and outputs untouched.  A state must not be updated from
 * two threads at once.
 */
#ifndef SPEC_STEP_H
#define SPEC_STEP_H

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_STEP_MAX_WINDOW 64

typedef struct {
    int32_t k_min;             /* smallest candidate step count, >= 0              */
    int32_t k_max;             /* largest, k_min <= k_max <= 31                    */
    int32_t k_init;            /* step used until the first switch, in range       */
    int32_t window_size;       /* completed batches in the window, 1..64 (20)      */
    int32_t update_interval;   /* re-score every this many batches, >= 1 (5)       */
    double switch_min_gain;    /* relative gain to exceed for a switch, >= 0 (0.05) */
} spec_step_policy;

/* Bytes of the opaque controller state. */
SPEC_API size_t spec_step_state_bytes(void);

/* Initialise a state of at least spec_step_state_bytes() bytes (any
 * alignment of 8) with a policy; the window starts empty. */
SPEC_API int spec_step_init(void *state, size_t state_bytes, const spec_step_policy *policy);

/*
 * Record one completed batch and return the step for the next one.
 *   acc, ver   [k_max] the batch's own counters (not running totals):
 *              acc[j] = #(requests with accepted length > j),
 *              ver[j] = #(requests with draft length > j); 0 <= acc[j] <= ver[j].
 *   cost_ms    [k_max + 1] full-step cost of each k for the next batch, > 0
 *              or +inf (k not covered); entries outside [k_min, k_max] are
 *              ignored.  Read only when a re-scoring is due.
 *   B          requests of the next batch, > 0.
 *   k_next     out: the step for the next batch.
 * Every update_interval-th batch re-scores every candidate over the window
 * and switches when the gain rule holds.
 */
SPEC_API int spec_step_update(void *state, const int64_t *acc, const int64_t *ver,
                              const double *cost_ms, int32_t B, int32_t *k_next);

/*
 * The last re-scoring: prefix_acceptance [k_max] (window values and the
 * extrapolated tail), score [k_max + 1] (0 outside [k_min, k_max] and for
 * infeasible k; all 0 before the first re-scoring with data), and the
 * current step.  Any output may be NULL.
 */
SPEC_API int spec_step_query(const void *state, double *prefix_acceptance, double *score,
                             int32_t *k_current);

/*
 * SPS cost model: n captured target graph sizes g_rows[i] (strictly
 * increasing, > 0) with measured full steps per second sps[i] > 0.
 * cost_ms[k] = 1000 / sps[i] for the first g_rows[i] >= B * (k + 1), +inf when
 * no captured size covers it; k = 0 .. k_max.
 */
SPEC_API int spec_step_cost_sps(int32_t B, int32_t k_max, const int32_t *g_rows,
                                const double *sps, int32_t n, double *cost_ms);

/*
 * Additive cost model: cost_ms[k] = 1000 * (bias_s + alpha_s[ib] + theta_s[ig])
 * with ib the first request bucket b_buckets[ib] >= B and ig the first graph
 * size g_rows[ig] >= B * (k + 1) (both lists strictly increasing, > 0);
 * +inf when either is not covered.  The terms are seconds and finite.
 */
SPEC_API int spec_step_cost_additive(int32_t B, int32_t k_max, double bias_s,
                                     const int32_t *b_buckets, const double *alpha_s, int32_t nb,
                                     const int32_t *g_rows, const double *theta_s, int32_t ng,
                                     double *cost_ms);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_STEP_H */
