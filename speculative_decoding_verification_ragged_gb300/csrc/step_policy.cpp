// Adaptive draft-step controller (host code): xLLM docs "自适应投机推理",
// §"自适应 draft 步长（MTP）" (one k per batch maximising
// B * (1 + sum_{j<k} prefix_acceptance[j]) / cost_ms(k)), §"可选的步长配置文件"
// (window of completed batches, re-scoring interval, minimum switch gain),
// §"成本模型与覆盖范围" (SPS and additive full-step cost over captured request
// and graph buckets).  The readings taken where the page is silent are listed
// in include/spec_step.h.
//
// The state lives in caller memory: the policy, a ring of the last
// window_size batches' counters (acc, ver per position) and the last scores.
// Window sums are exact int64; prefix acceptance and scores are fp64.
#include <cmath>
#include <cstring>
#include <limits>

#include "spec_step.h"

namespace {

constexpr uint64_t kStateTag = 0x5045545343455053ull;   // identifies an initialised state
constexpr int kMaxK = 31;

struct StepState {
    uint64_t tag;
    spec_step_policy pol;
    int64_t seen;                 // batches recorded so far
    int32_t k_cur;
    int32_t scored;               // 1 once a re-scoring had data
    int64_t acc[SPEC_STEP_MAX_WINDOW][kMaxK];
    int64_t ver[SPEC_STEP_MAX_WINDOW][kMaxK];
    double pa[kMaxK];
    double score[kMaxK + 1];
};

bool policy_ok(const spec_step_policy &p)
{
    return p.k_min >= 0 && p.k_min <= p.k_max && p.k_max <= kMaxK && p.k_init >= p.k_min &&
           p.k_init <= p.k_max && p.window_size >= 1 && p.window_size <= SPEC_STEP_MAX_WINDOW &&
           p.update_interval >= 1 && p.switch_min_gain >= 0.0;
}

// counts of one batch: 0 <= acc[j] <= ver[j], neither increasing with j
bool batch_ok(const int64_t *acc, const int64_t *ver, int k_max)
{
    for (int j = 0; j < k_max; ++j) {
        if (acc[j] < 0 || acc[j] > ver[j]) return false;
        if (j > 0 && (acc[j] > acc[j - 1] || ver[j] > ver[j - 1])) return false;
    }
    return true;
}

// sizes strictly increasing and positive
bool sizes_ok(const int32_t *s, int32_t n)
{
    if (!s || n < 1) return false;
    for (int32_t i = 0; i < n; ++i)
        if (s[i] <= 0 || (i > 0 && s[i] <= s[i - 1])) return false;
    return true;
}

// index of the first size >= need, or -1
int first_cover(const int32_t *s, int32_t n, int64_t need)
{
    for (int32_t i = 0; i < n; ++i)
        if (static_cast<int64_t>(s[i]) >= need) return i;
    return -1;
}

void rescore(StepState &st, const double *cost_ms, int32_t B)
{
    const spec_step_policy &p = st.pol;
    const int n = static_cast<int>(st.seen < p.window_size ? st.seen : p.window_size);
    int64_t A[kMaxK] = {}, V[kMaxK] = {};
    for (int s = 0; s < n; ++s)
        for (int j = 0; j < p.k_max; ++j) {
            A[j] += st.acc[s][j];
            V[j] += st.ver[s][j];
        }
    int last = -1;                                   // last verified position
    for (int j = 0; j < p.k_max; ++j)
        if (V[j] > 0) last = j;
    if (last < 0) return;                            // nothing verified: keep k
    double pa[kMaxK] = {};
    for (int j = 0; j <= last; ++j) pa[j] = static_cast<double>(A[j]) / static_cast<double>(V[j]);
    double rate = (last == 0) ? pa[0] : (pa[last - 1] > 0.0 ? pa[last] / pa[last - 1] : 0.0);
    rate = rate < 0.0 ? 0.0 : (rate > 1.0 ? 1.0 : rate);
    for (int j = last + 1; j < p.k_max; ++j) pa[j] = pa[j - 1] * rate;

    double score[kMaxK + 1] = {};
    for (int k = p.k_min; k <= p.k_max; ++k) {
        if (std::isinf(cost_ms[k])) continue;        // not covered: infeasible
        double expected = 1.0;                       // tokens per request: the bonus
        for (int j = 0; j < k; ++j) expected += pa[j];
        score[k] = static_cast<double>(B) * expected / cost_ms[k];
    }
    int best = p.k_min;
    for (int k = p.k_min; k <= p.k_max; ++k)
        if (score[k] > score[best]) best = k;        // ties: the smaller k
    if (score[best] > (1.0 + p.switch_min_gain) * score[st.k_cur]) st.k_cur = best;
    std::memcpy(st.pa, pa, sizeof pa);
    std::memcpy(st.score, score, sizeof score);
    st.scored = 1;
}

StepState *state_of(void *s)
{
    StepState *st = static_cast<StepState *>(s);
    return (st && st->tag == kStateTag) ? st : nullptr;
}

}  // namespace

extern "C" {

size_t spec_step_state_bytes(void) { return sizeof(StepState); }

int spec_step_init(void *state, size_t state_bytes, const spec_step_policy *policy)
{
    if (!state || state_bytes < sizeof(StepState) || !policy || !policy_ok(*policy))
        return SPEC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(state) % alignof(StepState) != 0) return SPEC_ERR_INVALID_ARG;
    StepState *st = static_cast<StepState *>(state);
    std::memset(st, 0, sizeof(StepState));
    st->tag = kStateTag;
    st->pol = *policy;
    st->k_cur = policy->k_init;
    return SPEC_OK;
}

int spec_step_update(void *state, const int64_t *acc, const int64_t *ver, const double *cost_ms,
                     int32_t B, int32_t *k_next)
{
    StepState *st = state_of(state);
    if (!st || !k_next || B <= 0) return SPEC_ERR_INVALID_ARG;
    const spec_step_policy &p = st->pol;
    if (p.k_max > 0 && (!acc || !ver)) return SPEC_ERR_INVALID_ARG;
    if (!batch_ok(acc, ver, p.k_max)) return SPEC_ERR_INVALID_ARG;
    const bool due = (st->seen + 1) % p.update_interval == 0;
    if (due) {
        if (!cost_ms) return SPEC_ERR_INVALID_ARG;
        for (int k = p.k_min; k <= p.k_max; ++k)
            if (!(cost_ms[k] > 0.0)) return SPEC_ERR_INVALID_ARG;   // NaN, 0, negative
    }
    const int slot = static_cast<int>(st->seen % p.window_size);
    for (int j = 0; j < p.k_max; ++j) {
        st->acc[slot][j] = acc[j];
        st->ver[slot][j] = ver[j];
    }
    st->seen += 1;
    if (due) rescore(*st, cost_ms, B);
    *k_next = st->k_cur;
    return SPEC_OK;
}

int spec_step_query(const void *state, double *prefix_acceptance, double *score,
                    int32_t *k_current)
{
    const StepState *st = state_of(const_cast<void *>(state));
    if (!st) return SPEC_ERR_INVALID_ARG;
    if (prefix_acceptance) std::memcpy(prefix_acceptance, st->pa, sizeof(double) * st->pol.k_max);
    if (score) std::memcpy(score, st->score, sizeof(double) * (st->pol.k_max + 1));
    if (k_current) *k_current = st->k_cur;
    return SPEC_OK;
}

int spec_step_cost_sps(int32_t B, int32_t k_max, const int32_t *g_rows, const double *sps,
                       int32_t n, double *cost_ms)
{
    if (B <= 0 || k_max < 0 || k_max > kMaxK || !sizes_ok(g_rows, n) || !sps || !cost_ms)
        return SPEC_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (!(sps[i] > 0.0) || std::isinf(sps[i])) return SPEC_ERR_INVALID_ARG;
    for (int k = 0; k <= k_max; ++k) {
        const int i = first_cover(g_rows, n, static_cast<int64_t>(B) * (k + 1));
        cost_ms[k] = (i < 0) ? std::numeric_limits<double>::infinity() : 1000.0 / sps[i];
    }
    return SPEC_OK;
}

int spec_step_cost_additive(int32_t B, int32_t k_max, double bias_s, const int32_t *b_buckets,
                            const double *alpha_s, int32_t nb, const int32_t *g_rows,
                            const double *theta_s, int32_t ng, double *cost_ms)
{
    if (B <= 0 || k_max < 0 || k_max > kMaxK || !sizes_ok(b_buckets, nb) ||
        !sizes_ok(g_rows, ng) || !alpha_s || !theta_s || !cost_ms || !std::isfinite(bias_s))
        return SPEC_ERR_INVALID_ARG;
    for (int32_t i = 0; i < nb; ++i)
        if (!std::isfinite(alpha_s[i])) return SPEC_ERR_INVALID_ARG;
    for (int32_t i = 0; i < ng; ++i)
        if (!std::isfinite(theta_s[i])) return SPEC_ERR_INVALID_ARG;
    const int ib = first_cover(b_buckets, nb, B);
    for (int k = 0; k <= k_max; ++k) {
        const int ig = first_cover(g_rows, ng, static_cast<int64_t>(B) * (k + 1));
        cost_ms[k] = (ib < 0 || ig < 0) ? std::numeric_limits<double>::infinity()
                                        : 1000.0 * (bias_s + alpha_s[ib] + theta_s[ig]);
    }
    return SPEC_OK;
}

}  // extern "C"
