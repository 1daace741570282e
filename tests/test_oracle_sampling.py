"""Pins for the oracle's filtered sampler (A3), point-mass rejection chain
(A4), draft confidence and prefix allocation (A6, A7) and prefix-acceptance
counters (A8).

The filters are checked against textbook formulations enumerated on tiny
vocabularies; the sampler against the Gumbel-max identity by chi-square; the
chain against the closed-form joint law of (accepted length, emitted token);
the allocation against exhaustive search.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

import workloads as W
from tests import _brute

FILTER_GRID = [
    # (T, top_k, top_p, min_p)
    (1.0, 0, 1.0, 0.0), (1.0, 3, 1.0, 0.0), (0.5, 0, 0.9, 0.0), (1.0, 0, 1.0, 0.2),
    (1.0, 4, 0.7, 0.0), (0.7, 5, 0.8, 0.1), (2.0, 2, 0.5, 0.3), (1.0, 1, 1.0, 0.0),
    (1.0, 0, 1.0, 1.0), (0.3, 9, 0.99, 0.01), (1.5, 12, 0.6, 0.0),
]


def _tiny_rows(seed, n, V, levels=5):
    """Rows over a few integer levels (scaled) so tie groups are common."""
    rng = np.random.default_rng(seed)
    return (rng.integers(0, levels, size=(n, V)) * 0.75 - 1.0).astype(np.float64)


@pytest.mark.parametrize("T,top_k,top_p,min_p", FILTER_GRID)
def test_filters_match_textbook_definitions(orc, T, top_k, top_p, min_p):
    for z in _tiny_rows(int(T * 100) + top_k, 40, 10):
        keep, margin = orc.filter_row(z, T, top_k, top_p, min_p)
        expect = _brute.survivors(list(z), T, top_k, top_p, min_p)
        if margin > 1e-9:   # decisions exactly at a float boundary are excluded
            assert set(np.nonzero(keep)[0]) == expect, (z, keep, expect)
        assert keep[int(np.argmax(z))]     # the top group always survives


def test_filter_special_cases(orc):
    z = np.array([1.0, 4.0, 2.0, 4.0, 0.0])
    keep, _ = orc.filter_row(z, 1.0, 1, 1.0, 0.0)        # top_k = 1 -> max tie group
    assert keep.tolist() == [False, True, False, True, False]
    keep, _ = orc.filter_row(z, 0.8, 0, 1.0, 1.0)        # min_p = 1 -> max tie group
    assert keep.tolist() == [False, True, False, True, False]
    keep, _ = orc.filter_row(z, 1.0, 0, 1.0, 0.0)        # no filter
    assert keep.all()
    keep, _ = orc.filter_row(z, 1.0, 5, 1.0, 0.0)        # top_k >= V is off
    assert keep.all()
    keep, _ = orc.filter_row(z, 1.0, 0, 1e-6, 0.0)       # tiny top_p -> top group only
    assert keep.tolist() == [False, True, False, True, False]


def test_sample_temperature_zero_and_topk1_are_greedy(orc):
    rng = np.random.default_rng(0)
    for t in range(30):
        z = rng.standard_normal(200) * 3
        a = int(np.argmax(z))
        y, _, _, _ = orc.sample_row(z, 0.0, 0, 1.0, 0.0, seed=t, rid=1, pos=0, step=0)
        assert y == a
        y, _, _, _ = orc.sample_row(z, 1.3, 1, 0.9, 0.0, seed=t, rid=1, pos=0, step=0)
        assert y == a                                     # unique max


@pytest.mark.parametrize("T,top_k,top_p,min_p", [
    (1.0, 0, 1.0, 0.0), (0.5, 0, 1.0, 0.0), (1.0, 4, 1.0, 0.0),
    (1.0, 0, 0.8, 0.0), (0.7, 0, 1.0, 0.15), (1.0, 5, 0.9, 0.05),
])
def test_sampler_distribution_chi_square(orc, T, top_k, top_p, min_p):
    z = np.array([1.2, -0.3, 0.9, 2.0, 0.1, 1.2, -1.0, 0.5])
    p = _brute.filtered_probs(list(z), T, top_k, top_p, min_p)
    n = 24_000
    counts = np.zeros(len(z))
    for s in range(n):
        y, _, _, _ = orc.sample_row(z, T, top_k, top_p, min_p, seed=0x9E3779B97F4A7C15 * (s + 1),
                                    rid=s % 7, pos=s % 3, step=s // 21)
        counts[y] += 1
    assert (counts[p == 0] == 0).all()
    live = p > 0
    stat = scipy.stats.chisquare(counts[live], n * p[live])
    assert stat.pvalue > 1e-4, (counts, n * p)


def test_sampler_deterministic(orc):
    z = np.random.default_rng(5).standard_normal(1000) * 3
    a = [orc.sample_row(z, 1.0, 0, 0.9, 0.0, seed=77, rid=2, pos=1, step=3)[0] for _ in range(3)]
    assert len(set(a)) == 1
    b = {orc.sample_row(z, 1.0, 0, 1.0, 0.0, seed=s, rid=2, pos=1, step=3)[0] for s in range(20)}
    assert len(b) > 5


def _joint_law(P, d, k):
    """P(a = m, emitted = y) for a point-mass draft: prod_{j<m} P_j(d_j) *
    P_m(y) * [y != d_m when m < k]."""
    V = P.shape[1]
    law = {}
    for m in range(k + 1):
        pre = np.prod([P[j, d[j]] for j in range(m)])
        for y in range(V):
            if m < k and y == d[m]:
                continue
            law[(m, y)] = pre * P[m, y]
    return law


def test_rejection_chain_joint_law(orc):
    # one request, k = 2, V = 4: rows with different shapes
    z = np.array([[1.0, 0.2, -0.5, 0.4], [0.0, 1.5, 0.3, 0.3], [0.8, -0.2, 0.1, 0.9]],
                 dtype=np.float32)
    d = np.array([0, 1, -1], dtype=np.int32)
    T, tk, tp, mp = 0.8, 3, 0.95, 0.0
    P = np.stack([_brute.filtered_probs(list(z[j].astype(np.float64)), T, tk, tp, mp)
                  for j in range(3)])
    law = _joint_law(P, d, 2)
    n = 20_000
    counts = {key: 0 for key in law}
    for s in range(n):
        params = W.SampleParams(np.array([T], np.float32), np.array([tk], np.int32),
                                np.array([tp], np.float32), np.array([mp], np.float32),
                                np.array([1234567 + 7919 * s], np.uint64),
                                np.array([3], np.uint32), step=s)
        res = orc.verify_sample(z, "f32", 4, 1, 2, np.array([0, 3]), d, params)
        counts[(int(res.accepted_len[0]), int(res.next_token[0]))] += 1
    keys = [kk for kk in law if law[kk] > 0]
    obs = np.array([counts[kk] for kk in keys], dtype=float)
    exp = np.array([law[kk] for kk in keys]) * n
    assert sum(counts[kk] for kk in law if law[kk] == 0) == 0
    assert scipy.stats.chisquare(obs, exp).pvalue > 1e-4
    # acceptance of the first draft is exactly P_0(d_0)
    acc0 = sum(v for (m, _), v in counts.items() if m >= 1) / n
    assert abs(acc0 - P[0, 0]) < 4 * math.sqrt(P[0, 0] * (1 - P[0, 0]) / n)


def test_sample_temperature_zero_equals_greedy_batch(orc):
    vb = W.ragged_batch(21, B=10, k_max=5, V=900, dtype="bf16", tie_top=True)
    params = W.SampleParams(np.zeros(10, np.float32), np.full(10, 20, np.int32),
                            np.full(10, 0.9, np.float32), np.full(10, 0.05, np.float32),
                            np.arange(10, dtype=np.uint64), np.arange(10, dtype=np.uint32))
    s = orc.verify_sample(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids,
                          params)
    g = orc.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    np.testing.assert_array_equal(s.out_tokens, g.out_tokens)
    np.testing.assert_array_equal(s.accepted_len, g.accepted_len)


def test_sample_bad_params_fall_back(orc):
    vb = W.ragged_batch(2, B=4, k_max=2, V=64, dtype="f32", k_values=np.array([2, 2, 2, 2]))
    params = W.SampleParams(np.array([-1.0, 1.0, 1.0, 1.0], np.float32),
                            np.array([0, -3, 0, 0], np.int32),
                            np.array([1.0, 1.0, 1.5, 1.0], np.float32),
                            np.array([0.0, 0.0, 0.0, -0.1], np.float32),
                            np.arange(4, dtype=np.uint64), np.arange(4, dtype=np.uint32))
    res = orc.verify_sample(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                            vb.draft_ids, params)
    assert res.status == (orc.BAD_TEMPERATURE | orc.BAD_TOP_K | orc.BAD_TOP_P | orc.BAD_MIN_P)
    g = orc.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    assert res.out_tokens[0].tolist() == g.out_tokens[0].tolist()   # bad T -> greedy


# ------------------------------------------------------ A6/A7 confidence -----

def test_confidence_closed_forms(orc):
    V, L = 500, 5.0
    uni = np.zeros((1, V), np.float32)
    one = np.zeros((1, V), np.float32)
    one[0, 123] = L
    x = np.concatenate([uni, one])
    a = orc.draft_confidence(x, "f32", V, 1, 2, threshold=0.0)
    assert a.conf[0] == pytest.approx(1.0 / V, rel=1e-13)           # argmax 0 of a flat row
    assert a.conf[1] == pytest.approx(math.exp(L) / (math.exp(L) + V - 1), rel=1e-13)


def test_confidence_matches_softmax(orc):
    db = W.mtp_adaptive(seed=3, B=3, k=4, V=2000, planted_draft=True)
    sel = np.random.default_rng(0).integers(0, 2000, size=12).astype(np.int32)
    a = orc.draft_confidence(db.draft_logits, "bf16", 2000, 3, 4, selected=sel, threshold=0.3)
    vals = W.bf16_bits_to_f32(db.draft_logits).astype(np.float64)
    p = scipy.special.softmax(vals, axis=1)
    np.testing.assert_allclose(a.conf, p[np.arange(12), sel], rtol=1e-12)


def test_allocation_extremes_and_packing(orc):
    db = W.mtp_adaptive(seed=5, B=4, k=3, V=300, planted_draft=True)
    a = orc.draft_confidence(db.draft_logits, "bf16", 300, 4, 3, threshold=0.0)
    assert a.k_alloc.tolist() == [3] * 4
    assert a.cu_rows.tolist() == [0, 4, 8, 12, 16] and a.total_rows == 16
    a = orc.draft_confidence(db.draft_logits, "bf16", 300, 4, 3, threshold=1.5)
    assert a.k_alloc.tolist() == [0] * 4 and a.total_rows == 4
    assert a.row_owner.tolist()[:4] == [0, 1, 2, 3] and (a.row_owner[4:] == -1).all()
    a = orc.draft_confidence(db.draft_logits, "bf16", 300, 4, 3, threshold=0.3)
    vals = W.bf16_bits_to_f32(db.draft_logits)
    top = np.argmax(vals, axis=1)
    for b in range(4):
        c = np.cumprod(a.conf[b * 3:(b + 1) * 3])
        assert a.k_alloc[b] == int((c >= 0.3).sum())
        for j in range(a.k_alloc[b] + 1):
            r = a.cu_rows[b] + j
            assert a.row_owner[r] == b and a.row_pos[r] == j
            assert a.packed_draft[r] == (top[b * 3 + j] if j < a.k_alloc[b] else -1)


@pytest.mark.parametrize("seed", range(6))
def test_allocation_budget_is_optimal(orc, seed):
    B, k = 3, 3
    db = W.mtp_adaptive(seed=seed, B=B, k=k, V=64, planted_draft=True)
    free = orc.draft_confidence(db.draft_logits, "bf16", 64, B, k, threshold=0.05)
    cum = np.concatenate([np.cumprod(free.conf[b * k:(b + 1) * k]) for b in range(B)])
    for G in range(B, B * (k + 1) + 1):
        a = orc.draft_confidence(db.draft_logits, "bf16", 64, B, k, threshold=0.05, max_rows=G)
        assert a.total_rows <= max(G, B) and (a.k_alloc <= free.k_alloc).all()
        got = sum(cum[b * k + j] for b in range(B) for j in range(a.k_alloc[b]))
        best = _brute.best_allocation(cum, B, k, list(free.k_alloc), G - B)
        assert got == pytest.approx(best, rel=1e-12)
    bad = orc.draft_confidence(db.draft_logits, "bf16", 64, B, k, threshold=0.0, max_rows=B - 1)
    assert bad.status & orc.BAD_BUDGET


# ------------------------------------------------------------ A8 counters -----

def test_prefix_stats_invariants_and_sharding(orc):
    vb = W.ragged_batch(4, B=40, k_max=6, V=50, dtype="f32", p_top=0.7)
    res = orc.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    acc, ver, hist, st = orc.prefix_stats(res.accepted_len, vb.cu_rows, vb.B, vb.k_max)
    assert st == 0
    kb = np.diff(vb.cu_rows) - 1
    assert acc.sum() == res.accepted_len.sum()
    assert (np.diff(acc) <= 0).all() and (np.diff(ver) <= 0).all() and (acc <= ver).all()
    assert ver.tolist() == [int((kb > j).sum()) for j in range(vb.k_max)]
    assert hist.sum() == vb.B and hist.tolist() == np.bincount(res.accepted_len,
                                                               minlength=vb.k_max + 1).tolist()
    # counters from a split batch sum to the unsplit counters
    cut = 17
    cu_a = vb.cu_rows[:cut + 1]
    cu_b = vb.cu_rows[cut:] - vb.cu_rows[cut]
    a1, v1, h1, _ = orc.prefix_stats(res.accepted_len[:cut], cu_a, cut, vb.k_max)
    a2, v2, h2, _ = orc.prefix_stats(res.accepted_len[cut:], cu_b, vb.B - cut, vb.k_max)
    assert (a1 + a2).tolist() == acc.tolist() and (v1 + v2).tolist() == ver.tolist()
    assert (h1 + h2).tolist() == hist.tolist()


def test_prefix_acceptance_matches_position_probabilities(orc):
    p = (0.9, 0.7, 0.5, 0.6)
    acc = ver = None
    for step in range(3):
        vb = W.planted_greedy(seed=500 + step, B=1500, k=4, V=48, p_pos=p, dtype="f32")
        res = orc.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                vb.draft_ids)
        acc, ver, _, _ = orc.prefix_stats(res.accepted_len, vb.cu_rows, vb.B, vb.k_max, acc, ver)
    rate = acc / ver
    expect = np.cumprod(p)
    assert np.all(np.abs(rate - expect) < 4 * np.sqrt(expect * (1 - expect) / ver))
