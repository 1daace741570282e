"""Independent brute-force formulations used to pin the oracle on tiny inputs.

Each function states the *textbook* form of a definition, which differs from
the form the oracle implements (rank counts vs. threshold enumeration,
logit-ratio vs. explicit probabilities, strict-mass rule vs. smallest
nucleus, greedy top-(G-B) vs. exhaustive search).  Pure Python; small V only.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
from scipy.special import softmax


def topk_set(z, k):
    """Top-k as the smallest upper set (whole tie groups) holding >= k tokens."""
    V = len(z)
    if k <= 0 or k >= V:
        return set(range(V))
    for t in sorted(set(z), reverse=True):
        up = {i for i in range(V) if z[i] >= t}
        if len(up) >= k:
            return up
    return set(range(V))


def minp_set(z, T, min_p):
    """Min-p with explicit probabilities: keep p_i >= min_p * max_j p_j."""
    V = len(z)
    if min_p <= 0:
        return set(range(V))
    p = softmax(np.asarray(z, dtype=np.float64) / T)
    pmax = p.max()
    return {i for i in range(V) if p[i] >= min_p * pmax}


def nucleus(z, T, top_p, allowed):
    """Top-p as the smallest upper set of `allowed` (whole tie groups) whose
    renormalised probability reaches top_p."""
    allowed = sorted(allowed)
    if top_p >= 1.0 or not allowed:
        return set(allowed)
    zz = np.asarray([z[i] for i in allowed], dtype=np.float64)
    p = softmax(zz / T)
    prob = dict(zip(allowed, p))
    for t in sorted({z[i] for i in allowed}, reverse=True):
        up = {i for i in allowed if z[i] >= t}
        if sum(prob[i] for i in up) >= top_p:
            return up
    return set(allowed)


def survivors(z, T, top_k, top_p, min_p):
    s = topk_set(z, top_k) & minp_set(z, T, min_p)
    return nucleus(z, T, top_p, s)


def filtered_probs(z, T, top_k, top_p, min_p):
    """Target distribution after filtering: softmax(z/T) restricted to the
    survivors and renormalised."""
    F = sorted(survivors(z, T, top_k, top_p, min_p))
    p = np.zeros(len(z))
    w = softmax(np.asarray([z[i] for i in F], dtype=np.float64) / T)
    p[F] = w
    return p


def best_allocation(cum, B, k, k_unbudgeted, budget):
    """Exhaustive search: prefix-closed allocations k_b <= k_unbudgeted[b]
    with sum(k_b) <= budget, maximising the summed cumulative confidence.
    Returns the optimum value."""
    best = -1.0
    for ks in itertools.product(*[range(kb + 1) for kb in k_unbudgeted]):
        if sum(ks) > budget:
            continue
        v = sum(cum[b * k + j] for b in range(B) for j in range(ks[b]))
        best = max(best, v)
    return best


def draft_rank(z, d):
    """Rank of token d by a descending sort: how many values lie strictly above."""
    s = np.sort(np.asarray(z, dtype=np.float64))[::-1]
    return int(np.searchsorted(-s, -z[d], side="left"))


def lse_direct(z):
    """log(sum(exp(z))) summed with math.fsum (exact rounding of the sum)."""
    m = max(z)
    if m == -math.inf:
        return -math.inf
    return m + math.log(math.fsum(math.exp(v - m) for v in z))
