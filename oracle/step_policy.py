"""Plain Python oracle of the adaptive draft-step controller.

TEST INFRASTRUCTURE ONLY: only the test-suite may use it.  It shares no code
with the library's controller; both are written separately from the same
definitions.

Source: xLLM docs "自适应投机推理" (adaptive speculative inference):
  §"自适应 draft 步长（MTP）" -- one step count k for the whole batch,
    maximising B * (1 + sum(prefix_acceptance[:k])) / cost_ms(k) over the
    candidates, from per-position prefix acceptance of completed batches;
  §"可选的步长配置文件" -- a window of completed batches (20), re-scoring
    every update_interval batches (5), a switch only when the predicted
    relative gain strictly exceeds switch_min_gain (0.05);
  §"成本模型与覆盖范围" -- full-step cost 1000 / SPS(G) ms, or the additive
    fit bias + alpha(Bcap) + theta(G) seconds; G is the first captured graph
    size covering the verified rows, B * (k + 1).

Readings where the page is silent (the same in the library):
  - prefix acceptance of position j = window sum of acc[j] / window sum of
    ver[j] (acc[j] = #(accepted > j), ver[j] = #(drafted > j));
  - positions never verified in the window continue with the conditional
    acceptance of the last verified one, pa[L] / pa[L-1] (pa[0] if L = 0),
    clamped to [0, 1];
  - ties in score go to the smaller k; an infeasible k (cost +inf) scores 0;
  - an empty window keeps the current k.
"""
import math


def _first_cover(sizes, need):
    for i, s in enumerate(sizes):
        if s >= need:
            return i
    return None


def _check_sizes(sizes):
    if len(sizes) == 0 or any(s <= 0 for s in sizes):
        raise ValueError("sizes must be positive")
    if any(b <= a for a, b in zip(sizes, sizes[1:])):
        raise ValueError("sizes must be strictly increasing")


def step_cost_sps(B, k_max, g_rows, sps):
    """cost_ms[k] = 1000 / SPS(G_k), G_k the first captured size >= B (k + 1)."""
    if B <= 0 or not (0 <= k_max <= 31) or len(g_rows) != len(sps):
        raise ValueError("bad arguments")
    _check_sizes(g_rows)
    if any(not (s > 0) or math.isinf(s) for s in sps):
        raise ValueError("sps must be positive and finite")
    out = []
    for k in range(k_max + 1):
        i = _first_cover(g_rows, B * (k + 1))
        out.append(math.inf if i is None else 1000.0 / sps[i])
    return out


def step_cost_additive(B, k_max, bias_s, b_buckets, alpha_s, g_rows, theta_s):
    """cost_ms[k] = 1000 (bias + alpha(Bcap) + theta(G_k)) with Bcap the first
    request bucket >= B and G_k the first graph size >= B (k + 1)."""
    if B <= 0 or not (0 <= k_max <= 31) or len(b_buckets) != len(alpha_s) \
            or len(g_rows) != len(theta_s):
        raise ValueError("bad arguments")
    _check_sizes(b_buckets)
    _check_sizes(g_rows)
    if not all(math.isfinite(x) for x in [bias_s, *alpha_s, *theta_s]):
        raise ValueError("terms must be finite")
    ib = _first_cover(b_buckets, B)
    out = []
    for k in range(k_max + 1):
        ig = _first_cover(g_rows, B * (k + 1))
        if ib is None or ig is None:
            out.append(math.inf)
        else:
            out.append(1000.0 * (bias_s + alpha_s[ib] + theta_s[ig]))
    return out


class StepController:
    """One k per batch from the window's prefix acceptance and the costs."""

    def __init__(self, k_min, k_max, k_init, window_size=20, update_interval=5,
                 switch_min_gain=0.05):
        if not (0 <= k_min <= k_max <= 31) or not (k_min <= k_init <= k_max):
            raise ValueError("bad step range")
        if not (1 <= window_size <= 64) or update_interval < 1 or not (switch_min_gain >= 0):
            raise ValueError("bad policy")
        self.k_min, self.k_max, self.k = k_min, k_max, k_init
        self.window_size, self.update_interval = window_size, update_interval
        self.gain = switch_min_gain
        self.batches = []
        self.prefix_acceptance = [0.0] * k_max
        self.score = [0.0] * (k_max + 1)

    def update(self, acc, ver, cost_ms, B):
        acc, ver = [int(x) for x in acc], [int(x) for x in ver]
        if len(acc) != self.k_max or len(ver) != self.k_max or B <= 0:
            raise ValueError("bad batch")
        for j in range(self.k_max):
            if not (0 <= acc[j] <= ver[j]):
                raise ValueError("need 0 <= acc <= ver")
            if j and (acc[j] > acc[j - 1] or ver[j] > ver[j - 1]):
                raise ValueError("counters must not increase with the position")
        due = (len(self.batches) + 1) % self.update_interval == 0
        if due:
            for k in range(self.k_min, self.k_max + 1):
                c = cost_ms[k]
                if math.isnan(c) or c <= 0:
                    raise ValueError("cost must be positive or +inf")
        self.batches.append((acc, ver))
        if due:
            self._rescore(cost_ms, B)
        return self.k

    def _rescore(self, cost_ms, B):
        window = self.batches[-self.window_size:]
        A = [sum(a[j] for a, _ in window) for j in range(self.k_max)]
        V = [sum(v[j] for _, v in window) for j in range(self.k_max)]
        seen = [j for j in range(self.k_max) if V[j] > 0]
        if not seen:
            return
        L = seen[-1]
        pa = [A[j] / V[j] if j <= L else 0.0 for j in range(self.k_max)]
        if L == 0:
            rate = pa[0]
        elif pa[L - 1] > 0:
            rate = pa[L] / pa[L - 1]
        else:
            rate = 0.0
        rate = min(max(rate, 0.0), 1.0)
        for j in range(L + 1, self.k_max):
            pa[j] = pa[j - 1] * rate
        score = [0.0] * (self.k_max + 1)
        for k in range(self.k_min, self.k_max + 1):
            if math.isinf(cost_ms[k]):
                continue
            expected = 1.0
            for j in range(k):
                expected += pa[j]
            score[k] = B * expected / cost_ms[k]
        best = self.k_min
        for k in range(self.k_min, self.k_max + 1):
            if score[k] > score[best]:
                best = k
        if score[best] > (1.0 + self.gain) * score[self.k]:
            self.k = best
        self.prefix_acceptance, self.score = pa, score
